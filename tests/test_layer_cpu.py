"""Host logic of the weight workspace (no GPU): an entry is reused while the
weight is the same storage, version, shape and quantizer role, and recast
into its own buffers otherwise (jax-aiter README, "Supported ops" row
"MXFP4 Quantizer / Workspace": quantized weights cached by name)."""
import torch

from quantization_mxfp4_cast_gb300.layer import MXFP4Quantizer, WeightWorkspace


class CountingQuantizer(MXFP4Quantizer):
    def __init__(self, role="weight", hadamard_col=False):
        super().__init__(role, hadamard_col)
        self.calls = []

    def quantize(self, t, out=None):
        self.calls.append((t.data_ptr(), t._version, out is not None))
        return out if out is not None else object()


def test_reuse_and_invalidation():
    ws = WeightWorkspace()
    q = CountingQuantizer()
    w = torch.zeros(64, 32)
    a = ws.get_or_quantize(w, q, "w")
    b = ws.get_or_quantize(w, q, "w")
    assert a is b and len(q.calls) == 1 and ws.casts == 1
    w.add_(1.0)                                # in-place update: new version
    c = ws.get_or_quantize(w, q, "w")
    assert len(q.calls) == 2 and q.calls[-1][2]  # recast into the entry's buffers
    assert c is a
    w2 = torch.zeros(64, 32)                   # other storage under the same name
    ws.get_or_quantize(w2, q, "w")
    assert len(q.calls) == 3
    ws.get_or_quantize(w2, q, "other")         # separate name, separate entry
    assert len(q.calls) == 4
    ws.get_or_quantize(w2, CountingQuantizer("activation", True), "other")  # other role
    assert ws.casts == 5
    ws.invalidate("other")
    ws.get_or_quantize(w2, q, "other")
    assert ws.casts == 6
    ws.invalidate()
    ws.get_or_quantize(w2, q, "w")
    assert ws.casts == 7


def test_presets():
    assert not MXFP4Quantizer.for_weight().hadamard_col
    assert MXFP4Quantizer.for_activation().hadamard_col
    assert MXFP4Quantizer.for_grad().hadamard_col
    assert {MXFP4Quantizer.for_weight().role, MXFP4Quantizer.for_activation().role,
            MXFP4Quantizer.for_grad().role} == {"weight", "activation", "grad"}


def test_stack_shape_validation():
    import pytest
    from quantization_mxfp4_cast_gb300.layer import MXFP4LinearStack
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        MXFP4LinearStack([])
    with pytest.raises(ValueError):
        MXFP4LinearStack([bf(64, 32), bf(32, 96)])   # 96 inputs after 64 outputs
    with pytest.raises(ValueError):
        MXFP4LinearStack([bf(48, 32)])               # 48 is not a multiple of 32
    s = MXFP4LinearStack([bf(64, 32), bf(96, 64)])
    assert [tuple(p.shape) for p in s.weights] == [(64, 32), (96, 64)]
