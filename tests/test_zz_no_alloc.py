"""moe_permute_noalloc: the permute for callers that cannot allocate device
memory (a host that owns all device memory through its own pool, or a
latency-critical path that must not pay cudaMalloc's synchronisation). Its
scratch is a fixed array inside the library, so it takes no workspace.

Checked through the C ABI against moe_permute (the workspace variant) on two
calls in a row with different routings: the layout is integer work and the
gathered rows are copies, so both must match bit for bit. The second call
also shows that the shared scratch's leftovers from the first call do no
harm. This file is collected last so that a failure here never hides
another test's result.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else t.data_ptr()


def _outputs(R_cap, T, k, E, d, dev):
    return dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int64, device=dev),
                dst_row=torch.empty(T * k, dtype=torch.int32, device=dev),
                src_pair=torch.empty(R_cap, dtype=torch.int32, device=dev),
                xp=torch.zeros(R_cap, d, dtype=torch.bfloat16, device=dev))


def test_noalloc_permute_matches_workspace_permute_twice():
    from mixture_experts_routed_softmax_gb300 import _lib
    from mixture_experts_routed_softmax_gb300.build import build
    build()
    lib = _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream().cuda_stream
    gen = torch.Generator(device="cpu").manual_seed(7)
    for call, (T, k, E, d, align) in enumerate([(1000, 4, 32, 256, 16), (3000, 8, 128, 136, 128)]):
        R_cap = int(lib.moe_row_capacity(T, k, E, align))
        # a skewed routing with distinct experts per token
        scores = torch.rand(T, E, generator=gen) * torch.linspace(1.0, 3.0, E)
        idx = scores.topk(k, dim=1).indices.to(torch.int32).to(dev)
        x = torch.randn(T, d, generator=gen).to(torch.bfloat16).to(dev)
        ref = _outputs(R_cap, T, k, E, d, dev)
        ws_bytes = int(lib.moe_workspace_size(_lib.MOE_WS_PERMUTE, T, d, E, k, align))
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        _lib.call("moe_permute", _p(idx), T, k, E, 0, align, _p(x), d, R_cap, _p(ref["counts"]),
                  _p(ref["offsets"]), _p(ref["dst_row"]), _p(ref["src_pair"]), _p(ref["xp"]),
                  _p(ws), ws.numel(), stream)
        got = _outputs(R_cap, T, k, E, d, dev)
        _lib.call("moe_permute_noalloc", _p(idx), T, k, E, align, _p(x), d, R_cap,
                  _p(got["counts"]), _p(got["offsets"]), _p(got["dst_row"]),
                  _p(got["src_pair"]), _p(got["xp"]), stream)
        assert lib.moe_status(stream) == _lib.MOE_OK
        R_pad = int(ref["offsets"][-1])
        for name in ("counts", "offsets", "dst_row", "src_pair"):
            assert torch.equal(got[name], ref[name]), f"call {call}: {name}"
        assert torch.equal(got["xp"][:R_pad], ref["xp"][:R_pad]), f"call {call}: xp"
        assert int(got["counts"].sum()) == T * k


def test_noalloc_permute_rejects_problems_beyond_its_scratch():
    from mixture_experts_routed_softmax_gb300 import _lib
    from mixture_experts_routed_softmax_gb300.build import build
    build()
    lib = _lib.load()
    P = 0x1000   # never dereferenced: the size check returns first
    T, k, E, d, align = 200_000, 8, 64, 8, 16     # 1.6M pairs need ~6.4 MB of scratch
    R_cap = int(lib.moe_row_capacity(T, k, E, align))
    rc = lib.moe_permute_noalloc(P, T, k, E, align, P, d, R_cap, P, P, P, P, P, None)
    assert rc == _lib.MOE_ERR_UNSUPPORTED
