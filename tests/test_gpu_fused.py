"""Parity of the fused expert forward (moe_expert_fwd_fused: one persistent
launch that runs gate/up and the activation, then the down projection with
the pair's score, the down tiles waiting on the gate/up tiles of their rows)
with the float64 oracle, through the C ABI.

The permute's maps are exact; A and the scored Yp rows of every pair within
the rules of tests/harness.py (padding rows exactly 0);
y within 2e-2 x RMS plus bf16's half-ulp. Cases: several tiles in every
dimension, ragged d and f, skewed loads with empty experts, one token, wide
and maximal E with top-32, shared experts with the clamped SwiGLU; at full
size the Qwen3-30B-A3B-shaped and fine-grained 512-expert workloads, y
checked element-wise against the oracle evaluated expert by expert. The
fused A is also compared with the five-call forward's on the same routing.
"""
import numpy as np
import pytest
import torch

import workloads
from harness import assert_bf16_out_close, assert_mag_close, bf16_floor, magnitudes, to_np
from oracle import moe_oracle as mo
from oracle.streamed import stream_layer

pytestmark = pytest.mark.gpu

CASES = {
    # name: (T, d, f, E, k, S, align, act, zipf_s, tau)
    "tiny": (256, 128, 256, 8, 2, 0, 128, None, None, None),
    "ragged_a16": (300, 200, 136, 6, 2, 0, 16, None, None, None),
    "multi_tile": (520, 392, 520, 8, 3, 0, 128, None, None, None),
    "skewed_empty": (700, 264, 384, 16, 4, 0, 32, None, 1.2, 1.5),
    "one_token": (1, 128, 128, 8, 2, 0, 16, None, None, None),
    "wide_E": (256, 128, 64, 160, 6, 0, 16, None, 1.1, 0.8),
    "max_E_and_k": (96, 64, 64, 1024, 32, 0, 16, None, None, None),
    "shared2_clamped": (520, 392, 520, 8, 3, 2, 128, (1.0, 1.702, 1.0), None, None),
    "qwen_like_shared": (1024, 2048, 768, 128, 8, 1, 16, (7.0, 1.702, 1.0), None, None),
}


def _inputs(name, T, d, f, E, k, S, align, zipf, tau):
    """Inputs with E + S experts' weights; the router sees the first E."""
    wl = workloads.Workload(name, T=T, d=d, f=f, E=E + S, k=k, zipf_s=zipf, align=align)
    inp = workloads.generate(wl, tau=tau)
    inp["w_router"] = inp["w_router"][:, :E].contiguous()
    if inp.get("bias") is not None:
        inp["bias"] = inp["bias"][:E].contiguous()
    return inp


def _fused(layer, x, idx):
    b = layer.fused_buffers(x.shape[0])
    fi = torch.as_tensor(idx, dtype=torch.int32).cuda()
    layer.forward_fused(x, b, forced_idx=fi)
    assert layer.status() == 0
    return b, fi


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_forward_parity(name):
    from mixture_experts_routed_softmax_gb300.layer import MoELayer
    T, d, f, E, k, S, align, act, zipf, tau = CASES[name]
    inp = _inputs(name, T, d, f, E, k, S, align, zipf, tau)
    layer = MoELayer.from_inputs(inp, k, align, act=act)
    fw = mo.forward(inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                    inp["w_down"], k, act=act, shared=S)
    x = inp["x"].cuda()
    b, fi = _fused(layer, x, fw["idx"])
    maps = mo.permute_maps(fw["idx"], E, align, b.R_cap, shared=S)
    for key in ("counts", "offsets", "dst_row", "src_pair"):
        np.testing.assert_array_equal(to_np(getattr(b, key)), maps[key])
    R_pad = maps["R_pad"]
    dst = maps["dst_row"]
    pad = np.setdiff1d(np.arange(R_pad), dst)
    mag = magnitudes(inp, fw, None, k, act=act, shared=S)
    w = np.concatenate([fw["w"].reshape(-1)] + [np.ones(T)] * S)
    out = {}
    A = to_np(b.a[:R_pad])
    out["A"] = assert_mag_close("A", A[dst], fw["A"], mag["A"])
    assert np.all(A[pad] == 0), "A: padding rows not zero"
    Yp = to_np(b.yp[:R_pad])
    out["Yp"] = assert_mag_close("Yp (scored)", Yp[dst], w[:, None] * fw["Yu"],
                                 np.abs(w)[:, None] * mag["Yu"])
    assert np.all(Yp[pad] == 0), "Yp: padding rows not zero"
    out["y"] = assert_bf16_out_close("y", to_np(b.y), fw["y"])
    out["y_bf16_floor"] = bf16_floor(fw["y"])
    # the five-call forward on the same routing: the same A up to the order
    # of the tensor cores' fp32 sums (tile shapes differ)
    bs = layer.buffers(T, backward=False)
    layer.forward(x, bs, forced_idx=fi)
    assert layer.status() == 0
    da = (b.a[:R_pad].float() - bs.a[:R_pad].float()).abs().max().item()
    out["A_vs_five_call_maxabs"] = da
    assert da <= 2.0 ** -6 * max(bs.a[:R_pad].float().abs().max().item(), 1e-30)
    print(name, {k_: (round(v, 6) if isinstance(v, float) else v) for k_, v in out.items()})


@pytest.mark.parametrize("name", ["qwen3_30b", "fine512"])
def test_fused_forward_fullsize(name):
    """The workloads the fused forward is measured on, at full size: maps
    exact, padding rows zero, every element of y against the oracle."""
    from mixture_experts_routed_softmax_gb300.layer import MoELayer
    wl = workloads.CONFIGS[name]
    inp = workloads.generate(wl, with_dy=False)
    T, k, E = wl.T, wl.k, wl.E
    x64 = mo.as_f64(inp["x"])
    bias = None if inp["bias"] is None else mo.as_f64(inp["bias"])
    logits = mo.router_logits(x64, mo.as_f64(inp["w_router"]), bias)
    idx = mo.select_topk(logits, k)
    layer = MoELayer.from_inputs(inp, k, wl.align)
    x = inp["x"].cuda()
    b, _ = _fused(layer, x, idx)
    maps = mo.permute_maps(idx, E, wl.align, b.R_cap)
    for key in ("counts", "offsets", "dst_row", "src_pair"):
        np.testing.assert_array_equal(to_np(getattr(b, key)), maps[key])
    R_pad = maps["R_pad"]
    real = torch.zeros(R_pad, dtype=torch.bool, device="cuda")
    real[torch.as_tensor(maps["dst_row"]).cuda()] = True
    for nm in ("a", "yp"):
        assert torch.count_nonzero(getattr(b, nm)[:R_pad][~real]).item() == 0, f"{nm} padding"
    ref = stream_layer(inp, logits, idx, k, backward=False)
    err = assert_bf16_out_close("y", to_np(b.y), ref["y"])
    print(name, {"y": round(err, 6), "y_bf16_floor": round(bf16_floor(ref["y"]), 6)})
