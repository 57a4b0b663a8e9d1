"""The benchmark's two arms describe the same workload: the reference arm (the
oracle on the host cores) prints the `config` the GPU arm builds for the decode
layer, and both count the same algorithmic bytes.  Host only: one bounded
oracle sample (about a second), no device."""
import contextlib
import io
import json
import types

import bench
from gemm_zq_rmsnorm_gb300 import inputs


def _gpu_arm_config(name, layer_shapes, layers=1, extra=()):
    # the attributes the GPU arm's LayerWorkload passes to decode_config
    wl = types.SimpleNamespace(name=name, layer_shapes=list(layer_shapes), layers=layers, extra=list(extra),
                               R=bench.rotation_copies(layer_shapes, layers, extra), fused=True, prefetch=False)
    return bench.decode_config(wl.name, wl.layer_shapes, wl.layers, wl.extra, wl.R, wl.fused, wl.prefetch)


def test_reference_arm_prints_the_gpu_arms_config():
    args = types.SimpleNamespace(steps=1, warmup=0)   # one bounded oracle sample
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference"
    assert line["config"] == _gpu_arm_config("decode-27b-layer", inputs.LAYER_27B)


def test_decode_config_bytes_and_rotation():
    cfg = _gpu_arm_config("decode-27b-layer", inputs.LAYER_27B)
    assert cfg["algorithmic_bytes_per_step"] == int(bench.layer_algo_bytes(inputs.LAYER_27B, 1))
    # the 27B-class layer holds 183 MiB of Q4_K: three copies exceed three times the 129 MB L2
    assert cfg["weight_copies_rotated"] == 3
    small = _gpu_arm_config("decode-small-28L+lm_head", inputs.SMALL_DECODE[:-1], 28, [inputs.SMALL_DECODE[-1]])
    assert small["projections"][-1].startswith("lm_head")
    assert small["hidden"] == 1024
