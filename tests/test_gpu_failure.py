"""Failure detection on the GPU without a GPU fault: a kernel whose bounded
wait runs out (its producer held on a flag that nothing sets) must give up,
record CP_ERR_DEVICE_TIMEOUT in the device status word that the host reads,
and leave the context usable for the next call."""
import numpy as np
import pytest
import torch

import oracle as O
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

CP_ERR_DEVICE_TIMEOUT = 9


def test_bounded_wait_gives_up_and_reports(cuda_dev):
    assert F.cp_device_status() == 0
    g = torch.Generator().manual_seed(3)
    q, k, v = (torch.randn(1, 128, 1, 64, generator=g).to(torch.bfloat16).to(cuda_dev) for _ in range(3))
    pos = torch.arange(128, dtype=torch.int32, device=cuda_dev)
    o = torch.full((1, 128, 1, 64), 7.0, dtype=torch.float32, device=cuda_dev)
    lse = torch.full((1, 1, 128), 7.0, dtype=torch.float32, device=cuda_dev)
    F.cp_selftest_stalled_producer(q, k, v, pos, o, lse, 20_000_000)  # 20 ms limit
    torch.cuda.synchronize()
    assert F.cp_device_status() == CP_ERR_DEVICE_TIMEOUT      # read and cleared
    assert F.cp_device_status() == 0
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)    # nothing was written
    # the context is intact: the same problem runs normally afterwards
    o2, l2 = F.cp_attn_partial(q, k, v, pos, pos)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    o_ref, l_ref = O.attn_direct(f(q), f(k), f(v), np.arange(128), np.arange(128))
    assert np.max(np.abs(f(o2) - o_ref)) <= 2e-2
    assert np.max(np.abs(f(l2) - l_ref)) <= 1e-3
    assert F.cp_device_status() == 0


def test_timeout_status_survives_until_read(cuda_dev):
    """Two timed-out launches, then one read: the word is sticky, not a count."""
    g = torch.Generator().manual_seed(4)
    q, k, v = (torch.randn(1, 128, 1, 64, generator=g).to(torch.bfloat16).to(cuda_dev) for _ in range(3))
    pos = torch.arange(128, dtype=torch.int32, device=cuda_dev)
    o = torch.empty((1, 128, 1, 64), dtype=torch.float32, device=cuda_dev)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device=cuda_dev)
    F.cp_selftest_stalled_producer(q, k, v, pos, o, lse, 5_000_000)
    F.cp_selftest_stalled_producer(q, k, v, pos, o, lse, 5_000_000)
    assert F.cp_device_status(clear=False) == CP_ERR_DEVICE_TIMEOUT
    assert F.cp_device_status() == CP_ERR_DEVICE_TIMEOUT
    assert F.cp_device_status() == 0


@pytest.mark.parametrize("kernel", [0, 1, 2], ids=["bf16_forward", "tf32_forward", "backward"])
def test_every_kernel_gives_up_a_stalled_wait(cuda_dev, kernel):
    """Each attention kernel's bounded waits: its producer held on a flag that
    nothing sets gives up after 10 ms, the status word reads
    CP_ERR_DEVICE_TIMEOUT (sticky until read), and the next call on the same
    context computes correctly (the backward's two launches both give up)."""
    assert F.cp_device_status() == 0
    F.cp_selftest_stalled_kernel(kernel, 10_000_000)
    torch.cuda.synchronize()
    assert F.cp_device_status() == CP_ERR_DEVICE_TIMEOUT
    assert F.cp_device_status() == 0
    g = torch.Generator().manual_seed(8)
    q, k, v, do = (torch.randn(1, 256, 2, 64, generator=g) for _ in range(4))
    pos = torch.arange(256, dtype=torch.int32, device=cuda_dev)
    f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    gp = np.arange(256)
    if kernel == 1:
        o, l = F.cp_attn_partial_f32(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev), pos, pos)
        o_ref, l_ref = O.attn_direct(f(q), f(k), f(v), gp, gp)
        assert np.max(np.abs(f(o) - o_ref)) <= 4e-3 and np.max(np.abs(f(l) - l_ref)) <= 2e-3
    else:
        qb, kb, vb, dob = (t.to(torch.bfloat16) for t in (q, k, v, do))
        o, l = F.cp_attn_partial(qb.to(cuda_dev), kb.to(cuda_dev), vb.to(cuda_dev), pos, pos)
        o_ref, l_ref = O.attn_direct(f(qb), f(kb), f(vb), gp, gp)
        assert np.max(np.abs(f(o) - o_ref)) <= 2e-2 and np.max(np.abs(f(l) - l_ref)) <= 1e-3
        if kernel == 2:
            dq, dk, dv = F.cp_attn_bwd_partial(qb.to(cuda_dev), kb.to(cuda_dev), vb.to(cuda_dev), o, dob.to(cuda_dev),
                                               l, pos, pos)
            ref = O.attn_bwd(f(qb), f(kb), f(vb), o_ref, f(dob), l_ref, gp, gp)
            for got, r in zip((dq, dk, dv), ref):
                assert np.max(np.abs(f(got) - r)) <= 1e-2 * np.max(np.abs(r))
    assert F.cp_device_status() == 0
