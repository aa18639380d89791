"""nsa_compress_kv_noalloc against nsa_compress_kv, through the C-ABI.

The allocation-free entry point serves callers that cannot allocate device
memory when they compress (a serving loop with a memory plan fixed up front,
an embedder that owns no device allocator).  It runs the same kernels with
the library's fixed scratch array instead of a workspace, so its output must
equal the workspace entry point's; two calls in a row check that what the
shared array keeps from one call does not leak into the next.  The file is
named so that pytest collects it last.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

from workloads import PREFILL_CONFIGS, decode_config, make_prefill, make_decode


def _pair(inp, B, T, H, G, dk, dv, layout, kk, vk):
    import sparse_attention_long_10_b300 as nsa
    phi = {k: inp[k].cuda() for k in ("pe_k", "pe_v", "w_k", "w_v")}
    k, v = inp[kk].cuda(), inp[vk].cuda()
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi)
    Nc = nsa.nsa_num_compressed(cfg)

    def buffers():
        return (torch.full((B, G, Nc, dk), float("nan"), dtype=torch.bfloat16, device="cuda"),
                torch.full((B, G, Nc, dv), float("nan"), dtype=torch.bfloat16, device="cuda"))

    kc_ref, vc_ref = buffers()
    ws = nsa.workspace(nsa.nsa_compress_workspace_size(cfg))
    nsa.nsa_compress_kv(cfg, layout, k, v, kc_ref, vc_ref, ws)
    outs = []
    assert nsa.nsa_device_status(ws) == 0
    for _ in range(2):                      # two calls in a row share the static scratch
        kc, vc = buffers()
        nsa.nsa_compress_kv_noalloc(cfg, layout, k, v, kc, vc)
        # the no-alloc call's own status word, in the fixed array
        assert nsa.nsa_compress_kv_noalloc_status() == 0
        outs.append((kc, vc))
    torch.cuda.synchronize()
    return (kc_ref, vc_ref), outs


@pytest.mark.parametrize("key,T", [("tiny_2k", None), ("prefill_8k", 2345)])
def test_noalloc_matches_workspace_entry_point_prefill_layout(key, T):
    import sparse_attention_long_10_b300 as nsa
    wl = PREFILL_CONFIGS[key]
    inp = make_prefill(wl, T=T)
    T = inp["q"].shape[1]
    ref, outs = _pair(inp, wl.B, T, wl.H, wl.G, wl.dk, wl.dv, nsa.NSA_LAYOUT_BTGD, "k", "v")
    for kc, vc in outs:
        # the same kernels in the same order: the compression tests' tolerance
        # is met with equality
        assert torch.equal(kc, ref[0]) and torch.equal(vc, ref[1])


def test_noalloc_matches_workspace_entry_point_decode_layout():
    import sparse_attention_long_10_b300 as nsa
    wl = decode_config()
    inp = make_decode(wl, B=2, T=3001)
    ref, outs = _pair(inp, 2, 3001, wl.H, wl.G, wl.dk, wl.dv, nsa.NSA_LAYOUT_BGTD, "kcache", "vcache")
    for kc, vc in outs:
        assert torch.equal(kc, ref[0]) and torch.equal(vc, ref[1])
