"""GPU parity of the writer, the decode schedule and the decode scorer against the oracle.

Every call goes through the C ABI (via the ctypes binding). Floating-point outputs are held to
|gpu - ref| <= 1e-4 * (1 + |ref|); quantised bytes and selected index sets are exact (the sets up
to keys tied with the k-th value within that tolerance).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import fp4_sparse_attention_mxfp4_gb300 as fx
from gpu_helpers import (DecodeRun, assert_cache_equal, assert_logits_close, assert_topk_match, bf16_dev, dev,
                         new_cache, oracle_cache)

pytestmark = pytest.mark.gpu


def _oracle_side(case):
    kv_p, kv_s = oracle_cache(case.layout.num_pages, case.k_bf16, case.all_slots())
    qp, qs = oracle.quantize_plain(case.q_bf16)
    return kv_p, kv_s, qp, qs


def _check_decode(run: DecodeRun, ref, rows=None, full_logits=True):
    case = run.case
    kv_p, kv_s, qp, qs = ref
    idx = run.topk_idx.cpu().numpy()
    val = run.topk_val.cpu().numpy()
    lg = run.logits.cpu().numpy() if run.logits is not None else None
    rows = range(case.batch) if rows is None else rows
    for b in rows:
        c = int(case.ctx_lens[b])
        ref_lg = oracle.row_logits(qp, qs, case.w, b, kv_p, kv_s, case.layout.block_tables[b], 0, c)
        if lg is not None and full_logits:
            assert_logits_close(lg[b, :c], ref_lg, f"{case.name} seq {b} logits")
        assert_topk_match(idx[b], val[b], ref_lg, case.topk, f"{case.name} seq {b}")
    assert int(run.status.item()) == 0, f"status {int(run.status.item()):#x}"


def test_writer_bytes_match_oracle():
    case = synth.decode_config(1)
    run = DecodeRun(case)
    torch.cuda.synchronize()
    kv_p, kv_s, qp, qs = _oracle_side(case)
    assert_cache_equal(run.kv_p, run.kv_s, kv_p, kv_s)
    assert np.array_equal(run.q_packed.cpu().numpy(), qp)
    assert np.array_equal(run.q_scale.cpu().numpy(), qs)


def test_writer_edge_values_and_skips():
    # Hand-built rows: exact grid points, every rounding midpoint, zeros, tiny and huge
    # magnitudes, subnormals, negative values rounding to -0; negative slots skipped.
    rng = synth.Rng(91)
    rows = []
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0,
                     -6.0, 0.0, -0.0, 0.1, -0.1, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 4.5, 5.5, -5.9, 5.99, 0.2, -0.01],
                    np.float32)
    for scale in (1.0, 2.0 ** -20, 2.0 ** 40, 2.0 ** -130, 2.0 ** 120):
        x = np.tile(mids, 4) * np.float32(scale)
        rows.append(x)
    rows.append(np.zeros(128, np.float32))
    rows.append(rng.normal(128).astype(np.float32) * 1e-38)
    for _ in range(9):
        rows.append((rng.normal(128) * np.exp(rng.normal(128) * 3)).astype(np.float32))
    x = synth.bf16_bits(np.stack(rows))
    T = x.shape[0]
    pages = 3
    slots = np.array([(i * 37) % (pages * 64) for i in range(T)], np.int32)
    slots[[2, 5, 11]] = -1
    kv_p, kv_s = new_cache(pages)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fx.idx_fp4_quant_and_cache(bf16_dev(x), dev(slots), kv_p, kv_s, status=status)
    torch.cuda.synchronize()
    ref_p, ref_s = oracle_cache(pages, x, slots)
    assert_cache_equal(kv_p, kv_s, ref_p, ref_s)
    assert int(status.item()) == 0
    # query path on the same rows, as one query row of 16 heads
    assert T == 16
    xq = x.reshape(1, 16, 128)
    qp = torch.empty((xq.shape[0], 16, 64), dtype=torch.uint8, device="cuda")
    qs = torch.empty((xq.shape[0], 16, 4), dtype=torch.uint8, device="cuda")
    fx.idx_fp4_quant_and_cache(bf16_dev(x[:0]), dev(np.zeros(0, np.int32)), kv_p, kv_s, q_bf16=bf16_dev(xq),
                               q_packed=qp, q_scale=qs)
    torch.cuda.synchronize()
    rp, rs = oracle.quantize_plain(xq)
    assert np.array_equal(qp.cpu().numpy(), rp)
    assert np.array_equal(qs.cpu().numpy(), rs)


def test_writer_flags_slot_past_pool():
    x = synth.qk_bf16(synth.Rng(92), (3,))
    kv_p, kv_s = new_cache(1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fx.idx_fp4_quant_and_cache(bf16_dev(x), dev(np.array([5, 64, 1000], np.int32)), kv_p, kv_s, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & fx.DEV_BAD_SLOT
    ref_p, ref_s = oracle_cache(1, x[:1], np.array([5], np.int32))
    assert_cache_equal(kv_p, kv_s, ref_p, ref_s)


@pytest.mark.parametrize("config", [1, 2])
def test_decode_small_configs(config):
    case = synth.decode_config(config)
    run = DecodeRun(case).run()
    ref = _oracle_side(case)
    assert_cache_equal(run.kv_p, run.kv_s, ref[0], ref[1])
    _check_decode(run, ref)


@pytest.mark.parametrize("heads", [16, 32, 64, 128])
def test_decode_heads_and_ragged_contexts(heads):
    ctx = [1, 63, 64, 65, 127, 128, 129, 300, 0, 1000, 2047, 2048, 2049, 5000]
    case = synth.decode_case(f"ragged_h{heads}", 100 + heads, ctx, heads, 2048 if heads != 16 else 64)
    run = DecodeRun(case).run()
    ref = _oracle_side(case)
    _check_decode(run, ref)


def test_decode_split_sequences_merge():
    # Enough keys that every sequence spans several CTAs and the candidate merge runs; topk
    # small and large relative to the per-CTA share.
    ctx = [200000, 3, 150001, 64, 99999]
    for k in (16, 2048):
        case = synth.decode_case(f"split_k{k}", 7 + k, ctx, 64, k)
        run = DecodeRun(case).run()
        ref = _oracle_side(case)
        _check_decode(run, ref)


def test_decode_many_rows_merge():
    # 16 split sequences, the merge's clusters all resident at once. Equal lengths keep every
    # CTA's share of a row in shared memory; one long sequence among short ones has ~130 lists,
    # more than the cluster stages, and is merged from global memory.
    cases = [synth.decode_case("rows16_even", 31, [20000] * 16, 64, 2048),
             synth.decode_case("rows16_long", 32, [200000] + [1500 + 97 * i for i in range(15)], 64, 2048)]
    for case in cases:
        run = DecodeRun(case).run()
        ref = _oracle_side(case)
        _check_decode(run, ref)


@pytest.mark.parametrize("n,n_x,topk", [(3000, 500, 2048), (60000, 0, 2048), (20000, 300, 64)])
def test_decode_exact_ties_lowest_index(n, n_x, topk):
    # One sequence whose keys are copies of two vectors (n_x of one at random places, the rest of
    # the other): its logits take two values, and the k-th key sits in a class of hundreds to
    # tens of thousands of exactly equal logits. Equal keys are taken in token order, so the
    # selection must be exactly the oracle's lowest indices. The sizes steer the merge through
    # each way of resolving the threshold bin: a few thousand tied candidates (radix levels on
    # the gathered bin), and more than the cluster can gather (levels through cluster sums, the
    # share read from global memory).
    case = synth.decode_case(f"ties_{n}_{n_x}_k{topk}", 60 + n_x, [n], 64, topk)
    order = np.argsort(synth.Rng(61).uniform(n), kind="stable")
    vx, vy = case.k_bf16[0].copy(), case.k_bf16[1].copy()
    case.k_bf16[:] = vy
    case.k_bf16[order[:n_x]] = vx
    run = DecodeRun(case).run()
    kv_p, kv_s, qp, qs = _oracle_side(case)
    ref = oracle.row_logits(qp, qs, case.w, 0, kv_p, kv_s, case.layout.block_tables[0], 0, n)
    vals = np.unique(ref)
    assert len(vals) <= 2
    if len(vals) == 2:
        assert vals[1] - vals[0] > 10 * 1e-4 * (1 + abs(vals[1])), "classes too close to order exactly"
    expect = np.sort(np.lexsort((np.arange(n), -ref))[:min(topk, n)])
    got = run.topk_idx.cpu().numpy()[0]
    assert np.array_equal(got[:len(expect)], expect), f"{int((got[:len(expect)] != expect).sum())} indices differ"
    assert_topk_match(got, run.topk_val.cpu().numpy()[0], ref, topk, case.name)
    assert int(run.status.item()) == 0


def test_decode_config3_full():
    case = synth.decode_config(3)
    run = DecodeRun(case).run()
    ref = _oracle_side(case)
    assert_cache_equal(run.kv_p, run.kv_s, ref[0], ref[1])
    _check_decode(run, ref)


@pytest.mark.parametrize("config", [4, 5])
def test_decode_full_size_sampled(config):
    """The long-context workloads at full size, in the benchmark's launch configuration: every
    logit of two sequences and of sampled keys of all sequences, and the top-k of two sequences."""
    case = synth.decode_config(config)
    run = DecodeRun(case).run()
    kv_p, kv_s, qp, qs = _oracle_side(case)
    lg = run.logits.cpu().numpy()
    rng = synth.Rng(1000 + config)
    for b in range(case.batch):
        c = int(case.ctx_lens[b])
        t = np.unique(np.concatenate([rng.integers(0, c - 1, 64), [0, c - 1]]))
        for t0 in t[:16]:
            ref = oracle.row_logits(qp, qs, case.w, b, kv_p, kv_s, case.layout.block_tables[b], int(t0), int(t0) + 1)
            assert_logits_close(lg[b, t0:t0 + 1], ref, f"seq {b} key {t0}")
    _check_decode(run, (kv_p, kv_s, qp, qs), rows=[0, case.batch - 1], full_logits=True)


def test_decode_without_debug_buffer_matches():
    case = synth.decode_config(2)
    a = DecodeRun(case).run()
    b = DecodeRun(case, debug_logits=False).run()
    assert torch.equal(a.topk_idx, b.topk_idx)
    assert torch.equal(a.topk_val, b.topk_val)


def test_decode_status_bad_page_and_ctx():
    case = synth.decode_case("badpage", 5, [300, 200], 16, 64)
    run = DecodeRun(case)
    run.bt[1, 1] = case.layout.num_pages + 5  # a page id outside the pool
    run.run()
    assert int(run.status.item()) & fx.DEV_BAD_PAGE
    run2 = DecodeRun(case, max_ctx=250)
    run2.run()
    assert int(run2.status.item()) & fx.DEV_BAD_CTX  # 300 > max_ctx: that sequence is treated as empty
    assert np.all(run2.topk_idx.cpu().numpy()[0] == -1)


def test_decode_schedule_mismatch_flagged():
    case = synth.decode_case("mismatch", 6, [300, 200, 100], 16, 64)
    run = DecodeRun(case)
    run.schedule()
    run.ctx = run.ctx[:2].contiguous()
    run.q_packed = run.q_packed[:2].contiguous()
    run.q_scale = run.q_scale[:2].contiguous()
    run.w = run.w[:2].contiguous()
    run.topk_idx = run.topk_idx[:2].contiguous()
    run.topk_val = run.topk_val[:2].contiguous()
    run.logits = run.logits[:2].contiguous()
    run.score()
    torch.cuda.synchronize()
    assert int(run.status.item()) & fx.DEV_BAD_SCHEDULE


def parse_decode_schedule(buf, max_batch):
    """The decode schedule's tables, read on the host (header, per-range first unit, per-sequence
    context / first segment / segment count, units, segments)."""
    s = buf.cpu().numpy().view(np.int32)
    keys = ["magic", "ctas", "batch", "max_batch", "next_n", "rounds", "per", "num_units", "num_segs", "units_cap",
            "segs_cap", "ranges_cap", "total_tiles", "tiles_cap", "ok", "aligned"]
    h = dict(zip(keys, (int(x) for x in s[:16])))
    o = 16
    range_first = s[o:o + h["ranges_cap"] + 1]
    o += h["ranges_cap"] + 1
    seq_ctx, seq_seg0, seq_nseg = (s[o + i * max_batch:o + (i + 1) * max_batch] for i in range(3))
    uoff = ((o + 3 * max_batch) * 4 + 31) // 32 * 32 // 4
    units = s[uoff:uoff + 8 * h["units_cap"]].reshape(-1, 8)
    segs = s[uoff + 8 * h["units_cap"]:uoff + 8 * (h["units_cap"] + h["segs_cap"])].reshape(-1, 8)
    return h, range_first, seq_ctx, seq_seg0, seq_nseg, units, segs


@pytest.mark.parametrize("nseq,next_n", [(8, 1), (40, 1), (8, 2), (40, 2), (40, 4)])
def test_decode_schedule_invariants(nseq, next_n):
    """Units of every sequence partition [0, ctx) exactly in token order; each CTA range holds at
    most one row buffer of tiles; segments group a sequence's units per round with consecutive unit
    indices; sequences without keys have no segment. With verify rows the ranges may be cut from
    the tiles padded to whole ranges per sequence (every sequence then starts a range)."""
    base = np.array([131072, 5, 0, 70000, 128, 129, 1, 262144], np.int32)
    extra = synth.Rng(77).integers(0, 9000, max(nseq - len(base), 0)).astype(np.int32)
    ctx = np.concatenate([base, extra])[:nseq]
    max_batch = 16 if nseq <= 16 else 64
    sched = torch.zeros(fx.idx_fp4_decode_schedule_bytes(max_batch, 262144), dtype=torch.uint8, device="cuda")
    if next_n == 1:
        fx.idx_fp4_build_decode_schedule(dev(ctx), max_batch, 262144, sched)
    else:
        fx.idx_fp4_build_decode_schedule_mtp(dev(ctx), next_n, max_batch, 262144, sched)
    torch.cuda.synchronize()
    h, range_first, seq_ctx, seq_seg0, seq_nseg, units, segs = parse_decode_schedule(sched, max_batch)
    assert h["magic"] == 0x44534333 and h["ok"] == 1 and h["batch"] == nseq and h["max_batch"] == max_batch
    assert h["ctas"] == torch.cuda.get_device_properties(0).multi_processor_count
    tiles = [-(-int(c) // 128) for c in ctx]
    assert h["total_tiles"] == sum(tiles)
    assert np.array_equal(seq_ctx[:nseq], ctx)
    per, ctas, rounds = h["per"], h["ctas"], h["rounds"]
    assert 1 <= per <= (128 if next_n <= 2 else 64) and rounds * ctas * per >= h["total_tiles"]
    assert h["aligned"] in ((0,) if next_n == 1 else (0, 1))
    starts = np.concatenate([[0], np.cumsum(tiles)])
    # the layout the ranges are cut from: tiles end to end, or padded to whole ranges
    padded = [-(-t // per) * per for t in tiles] if h["aligned"] else tiles
    vstarts = np.concatenate([[0], np.cumsum(padded)])
    assert vstarts[-1] <= rounds * ctas * per
    covered = {b: [] for b in range(nseq)}
    for i in range(rounds * ctas):
        lo = i * per
        for ui in range(range_first[i], range_first[i + 1]):
            seq, kb, ke, buf, seg, uidx, tile0 = units[ui][:7]
            covered[seq].append((kb, ke, ui, seg, uidx))
            assert tile0 == starts[seq] + kb // 128 and kb % 128 == 0
            vt0 = vstarts[seq] + kb // 128
            assert lo <= vt0 and vt0 + -(-(ke - kb) // 128) <= lo + per
            assert buf == (vt0 - lo) * 128 and buf + (ke - kb) <= per * 128
            if h["aligned"]:
                assert range_first[i + 1] - range_first[i] == 1 and buf == 0
    assert range_first[rounds * ctas] == h["num_units"]
    nsegs = 0
    for b in range(nseq):
        r = sorted(covered[b])
        if ctx[b] == 0:
            assert r == [] and seq_nseg[b] == 0
            continue
        assert r[0][0] == 0 and r[-1][1] == ctx[b]
        assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
        assert seq_nseg[b] >= 1
        for k in range(seq_nseg[b]):
            sid = seq_seg0[b] + k
            sseq, first, nunits, skb, ske, rank = segs[sid][:6]
            mine = [x for x in r if x[3] == sid]
            assert sseq == b and rank == k and nunits == len(mine) and first == mine[0][2]
            assert [x[4] for x in mine] == list(range(nunits))
            assert [x[2] for x in mine] == list(range(first, first + nunits))
            assert skb == mine[0][0] and ske == mine[-1][1]
        nsegs += int(seq_nseg[b])
    assert nsegs == h["num_segs"]


def test_decode_several_rounds():
    """More keys than one pass of the grid holds (a range is at most 16384 keys at next_n 1): the
    step runs in rounds, sequences cut by a round boundary are merged from their segments' lists.
    Rows of sequences on both sides of the boundary against the oracle, and the schedule's rounds."""
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 256)
    per_round = sms * 128 * 128
    nseq = -(-(per_round * 9 // 8) // 131072)
    ctx = [131072] * (nseq - 1) + [100003]
    case = synth.decode_case("rounds", 41, ctx, 64, 2048)
    run = DecodeRun(case).run()
    h = parse_decode_schedule(run.sched, run.max_batch)[0]
    assert h["rounds"] >= 2 and h["ok"] == 1
    boundary = min(h["ctas"] * h["per"] // 1024, nseq - 1)  # the sequence holding the first round's end
    ref = _oracle_side(case)
    _check_decode(run, ref, rows=[0, boundary, nseq - 1], full_logits=True)


def test_decode_forty_ragged_sequences():
    """40 short sequences of ragged lengths (one empty): every row against the oracle."""
    ctx = synth.Rng(78).integers(1, 6000, 40).astype(np.int32)
    ctx[3] = 0
    case = synth.decode_case("batch40", 79, ctx, 32, 256)
    run = DecodeRun(case).run()
    ref = _oracle_side(case)
    _check_decode(run, ref)
