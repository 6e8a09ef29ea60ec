"""Streams, CUDA graphs and concurrent host threads.

Every call is asynchronous on the stream it is given; the prefetch path of the
ring adds a pooled side stream joined back with events.  These tests check that
  * a ring captured in a CUDA graph (side stream included) and replayed on new
    inputs gives exactly the eager results, in every ring mode and with the work
    plan in the workspace;
  * the same call on a non-default stream gives exactly the default stream's
    results;
  * two host threads running prefetched rings at once on their own streams each
    get exactly their single-threaded results (no shared side stream or event).
"""
import threading

import pytest
import torch

import cp_synth as SY
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

CASES = {
    "s4k": SY.WORKLOADS["s4k"],
    # the plan in the workspace: its two pre-pass kernels are captured too
    "global_plan": SY.Workload("st_plan", B=1, S=32 * 4224, N=2, Nkv=1, D=64, C=32),
}


def _shards(w, dev, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda n: F.cp_zigzag_shard(torch.randn(w.B, w.S, n, w.D, generator=g).to(torch.bfloat16).to(dev), w.C)  # noqa: E731
    return mk(w.N), mk(w.Nkv), mk(w.Nkv)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("prefetch,fused", [(1, False), (1, True), (0, False)])
def test_ring_in_a_cuda_graph_matches_eager(cuda_dev, name, prefetch, fused):
    w = CASES[name]
    qs, ks, vs = _shards(w, cuda_dev, 1)
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    ws = torch.empty(max(256, F.cp_ring_workspace_size(w.B, w.S, w.N, w.Nkv, w.D, w.C, prefetch, F.CP_F32, fused)),
                     dtype=torch.uint8, device=cuda_dev)
    o = torch.empty((w.C, w.B, w.S // w.C, w.N, w.D), dtype=torch.float32, device=cuda_dev)
    lse = torch.empty((w.C, w.B, w.N, w.S // w.C), dtype=torch.float32, device=cuda_dev)

    def ring():
        F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=prefetch, fused_merge=fused, workspace=ws, o=o, lse=lse)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ring()  # warm-up outside the capture (lazy set-up of the side stream and kernel attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ring()
    for seed in (2, 3):
        q2, k2, v2 = _shards(w, cuda_dev, seed)
        qs.copy_(q2)
        ks.copy_(k2)
        vs.copy_(v2)
        graph.replay()
        torch.cuda.synchronize()
        o_g, l_g = o.clone(), lse.clone()
        o_e, l_e = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=prefetch, fused_merge=fused)
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e), seed
    assert F.cp_device_status() == 0


def test_non_default_stream_matches_default(cuda_dev):
    w = SY.WORKLOADS["s4k"]
    qs, ks, vs = _shards(w, cuda_dev, 4)
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    o_d, l_d = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o_s, l_s = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1, stream=s)
        o_u = F.cp_zigzag_unshard(o_s, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o_s, o_d) and torch.equal(l_s, l_d)
    assert torch.equal(o_u, F.cp_zigzag_unshard(o_d))


def test_two_host_threads_run_rings_at_once(cuda_dev):
    w = SY.WORKLOADS["s4k"]
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    inputs = [_shards(w, cuda_dev, 10 + i) for i in range(2)]
    ref = [F.cp_ring_attention_fwd(*x, pos, prefetch=1) for x in inputs]
    torch.cuda.synchronize()
    out, errs = [None, None], []

    def worker(i):
        try:
            torch.cuda.set_device(cuda_dev)
            s = torch.cuda.Stream()
            res = []
            with torch.cuda.stream(s):
                for _ in range(4):
                    res.append(F.cp_ring_attention_fwd(*inputs[i], pos, prefetch=1, stream=s))
            s.synchronize()
            out[i] = res
        except Exception as e:  # reported below
            errs.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errs, errs
    for i in range(2):
        assert out[i] is not None
        for o, l in out[i]:
            assert torch.equal(o, ref[i][0]) and torch.equal(l, ref[i][1])
    assert F.cp_device_status() == 0
