"""Failure detection on the GPU without a GPU fault.

Every device-side wait of the library is bounded (0.5 s): a wait that runs
out records NSA_ERR_DEVICE_TIMEOUT in the workspace status word, the CTA
drains its copies in flight and frees its tensor memory, and the context
stays usable.  The test hook NSA_FLAG_TEST_STALL makes the compression
kernel's first CTA withhold one pipeline stage (a signal that nothing sends),
so one such wait runs out; the next call on the same workspace must then run
clean and give the normal result."""
import pytest
import torch

pytestmark = pytest.mark.gpu

from workloads import PREFILL_CONFIGS, make_prefill


def test_bounded_wait_times_out_and_the_next_call_is_clean():
    import sparse_attention_long_10_b300 as nsa
    wl = PREFILL_CONFIGS["tiny_2k"]
    inp = make_prefill(wl)
    d = {k: v.cuda() for k, v in inp.items()}
    cfg = nsa.make_cfg(wl.B, wl.T, wl.H, wl.G, wl.dk, wl.dv, phi=d)
    Nc = nsa.nsa_num_compressed(cfg)
    shape_k, shape_v = (wl.B, wl.G, Nc, wl.dk), (wl.B, wl.G, Nc, wl.dv)
    ws = nsa.workspace(nsa.nsa_compress_workspace_size(cfg))
    ref_k = torch.empty(shape_k, dtype=torch.bfloat16, device="cuda")
    ref_v = torch.empty(shape_v, dtype=torch.bfloat16, device="cuda")
    nsa.nsa_compress_kv(cfg, nsa.NSA_LAYOUT_BTGD, d["k"], d["v"], ref_k, ref_v, ws)
    assert nsa.nsa_device_status(ws) == 0

    stalled = nsa.make_cfg(wl.B, wl.T, wl.H, wl.G, wl.dk, wl.dv, phi=d, flags=nsa.NSA_FLAG_TEST_STALL)
    kc = torch.zeros(shape_k, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros(shape_v, dtype=torch.bfloat16, device="cuda")
    nsa.nsa_compress_kv(stalled, nsa.NSA_LAYOUT_BTGD, d["k"], d["v"], kc, vc, ws)
    assert nsa.nsa_device_status(ws) == 6          # NSA_ERR_DEVICE_TIMEOUT, read and cleared
    assert nsa.nsa_device_status(ws) == 0

    # the context and the workspace are usable: a normal call gives the normal result
    kc2 = torch.full(shape_k, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc2 = torch.full(shape_v, float("nan"), dtype=torch.bfloat16, device="cuda")
    nsa.nsa_compress_kv(cfg, nsa.NSA_LAYOUT_BTGD, d["k"], d["v"], kc2, vc2, ws)
    assert nsa.nsa_device_status(ws) == 0
    assert torch.equal(kc2, ref_k) and torch.equal(vc2, ref_v)
