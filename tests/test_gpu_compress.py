"""GPU parity of nsa_compress_kv (tcgen05 GEMM) against the oracle's compress."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import nsa as O
from workloads import PREFILL_CONFIGS, decode_config, make_prefill, make_decode
from tests.gpu_util import bf16_compare, compress_exact


def _nsa():
    import sparse_attention_long_10_b300 as nsa
    return nsa


def _run(inp, B, T, H, G, dk, dv, layout):
    nsa = _nsa()
    phi = {k: inp[k].cuda() for k in ("pe_k", "pe_v", "w_k", "w_v")}
    kk, vv = ("k", "v") if layout == nsa.NSA_LAYOUT_BTGD else ("kcache", "vcache")
    k, v = inp[kk].cuda(), inp[vv].cuda()
    cfg = nsa.make_cfg(B, T, H, G, dk, dv, phi)
    Nc = nsa.nsa_num_compressed(cfg)
    kc = torch.full((B, G, Nc, dk), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full((B, G, Nc, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = nsa.workspace(nsa.nsa_compress_workspace_size(cfg))
    nsa.nsa_compress_kv(cfg, layout, k, v, kc, vc, ws)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(ws) == 0
    return kc, vc


def _exact(inp, B, G, layout_btgd, kname, pename, wname):
    return compress_exact(inp, B, G, layout_btgd, kname, pename, wname)


@pytest.mark.parametrize("key,T", [("tiny_2k", None), ("tiny_2k", 1000), ("tiny_2k", 47),
                                   ("prefill_8k", None), ("prefill_8k", 2345)])
def test_compress_prefill_layout(key, T):
    wl = PREFILL_CONFIGS[key]
    inp = make_prefill(wl, T=T)
    T = inp["q"].shape[1]
    nsa = _nsa()
    kc, vc = _run(inp, wl.B, T, wl.H, wl.G, wl.dk, wl.dv, nsa.NSA_LAYOUT_BTGD)
    nk = bf16_compare(kc, *_exact(inp, wl.B, wl.G, True, "k", "pe_k", "w_k"))
    nv = bf16_compare(vc, *_exact(inp, wl.B, wl.G, True, "v", "pe_v", "w_v"))
    print(f"T={T}: rounding flips k={nk} v={nv}")


def test_compress_decode_layout_ragged():
    wl = decode_config()
    inp = make_decode(wl, B=2, T=3001)
    nsa = _nsa()
    kc, vc = _run(inp, 2, 3001, wl.H, wl.G, wl.dk, wl.dv, nsa.NSA_LAYOUT_BGTD)
    bf16_compare(kc, *_exact(inp, 2, wl.G, False, "kcache", "pe_k", "w_k"))
    bf16_compare(vc, *_exact(inp, 2, wl.G, False, "vcache", "pe_v", "w_v"))


def test_compress_short_sequence_is_empty():
    wl = PREFILL_CONFIGS["tiny_2k"]
    inp = make_prefill(wl, T=31)
    nsa = _nsa()
    kc, vc = _run(inp, 1, 31, wl.H, wl.G, wl.dk, wl.dv, nsa.NSA_LAYOUT_BTGD)
    assert kc.numel() == 0 and vc.numel() == 0
