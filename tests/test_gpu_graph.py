"""CUDA-graph replay of the decode step ("Score a DSA sparse indexer in FP4": the schedule is built
once a step at a CUDAGraph-stable address, so a captured graph replays across changing context
lengths; replay is bitwise stable, including re-replaying the capture batch after the others).

The schedule build and the decode call are captured once on the maximum context set of the
16 x 131072 workload; the context vector is then rewritten in place and the graph replayed on
{max}, {U[65536, max]}, {U[1, max]} (some below k) and {max} again.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import DecodeRun, assert_topk_match, oracle_cache

pytestmark = pytest.mark.gpu


def test_graph_replay_across_context_sets():
    case = synth.decode_config(4)
    run = DecodeRun(case, max_batch=16, max_ctx=131072, debug_logits=False)
    torch.cuda.synchronize()
    sets = synth.replay_ctx_sets(3, case.batch, 131072)
    run.ctx.copy_(torch.from_numpy(sets[0]))
    # warm up outside capture, then capture schedule + decode
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run.schedule()
        run.score()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run.schedule()
        run.score()
    torch.cuda.synchronize()

    kv_p, kv_s = oracle_cache(case.layout.num_pages, case.k_bf16, case.all_slots())
    qp, qs = oracle.quantize_plain(case.q_bf16)
    outs = []
    for si, ctx in enumerate(sets):
        run.ctx.copy_(torch.from_numpy(ctx))
        run.topk_idx.fill_(-7)
        run.topk_val.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        idx, val = run.topk_idx.cpu().numpy().copy(), run.topk_val.cpu().numpy().copy()
        outs.append((idx, val))
        # the same set through direct calls gives the same bits
        run.schedule()
        run.score()
        torch.cuda.synchronize()
        assert np.array_equal(run.topk_idx.cpu().numpy(), idx)
        assert np.array_equal(run.topk_val.cpu().numpy().view(np.uint32), val.view(np.uint32))
        # oracle parity on two sequences of the set (the shortest and the longest)
        for b in {int(np.argmin(ctx)), int(np.argmax(ctx))}:
            c = int(ctx[b])
            ref = oracle.row_logits(qp, qs, case.w, b, kv_p, kv_s, case.layout.block_tables[b], 0, c)
            assert_topk_match(idx[b], val[b], ref, case.topk, f"set {si} seq {b} (ctx {c})")
    assert int(run.status.item()) == 0
    # re-replaying the capture set after the others is bitwise identical to its first replay
    assert np.array_equal(outs[0][0], outs[3][0])
    assert np.array_equal(outs[0][1].view(np.uint32), outs[3][1].view(np.uint32))
    assert np.any(sets[2] < case.topk), "the third set includes contexts shorter than k"
