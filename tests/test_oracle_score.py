"""Pins for the oracle's scoring, page walk, selection and padding rows (CPU only).

Independent anchors:
  * H = 1, w = 1 reduces the score to relu(q . k): a numpy dot product of the
    dequantised vectors;
  * brute force on tiny inputs through numpy einsum over a dense, unpaged key matrix;
  * exact rational arithmetic (fractions.Fraction) on a tiny case: the fp64 oracle
    must agree to rounding of the final head sum;
  * invariance of the paged walk under any permutation of the pool's pages, and the
    identity page table reducing to the flat layout;
  * top-k against numpy's lexsort (a library sort) on random and tie-heavy data;
  * a padding row (row_end 0, "PCP correctness fixes", section 3) reads no key: with
    NaN scale sentinels in key 0 and every unwritten row its output stays all -1 and
    the other rows stay finite.
"""
from fractions import Fraction

import numpy as np

import oracle
import synth


def _pool(num_pages):
    return (np.full((num_pages, 4, 64, 16), 0x77, np.uint8), np.full((num_pages, 4, 64), 0xFF, np.uint8))


def _decode_setup(seed, ctx_lens, H, spare=0.125):
    rng = synth.Rng(seed)
    lay = synth.paged_layout(rng.fork(1), ctx_lens, spare=spare)
    k = synth.qk_bf16(rng.fork(2), (int(np.sum(ctx_lens)),))
    q = synth.qk_bf16(rng.fork(3), (len(ctx_lens), H))
    w = synth.head_weights(rng.fork(4), len(ctx_lens), H)
    kv_p, kv_s = _pool(lay.num_pages)
    slots = np.concatenate([lay.slots(b, 0, c) for b, c in enumerate(ctx_lens)])
    assert oracle.quant_and_cache(k, slots, kv_p, kv_s) == len(slots)
    qp, qs = oracle.quantize_plain(q)
    return lay, k, q, w, kv_p, kv_s, qp, qs


def test_single_head_unit_weight_is_relu_dot():
    lay, k, q, w, kv_p, kv_s, qp, qs = _decode_setup(31, [150], 1)
    w1 = np.ones_like(w)
    lg = oracle.decode_logits(qp, qs, w1, kv_p, kv_s, lay.block_tables, np.array([150], np.int32))
    qd = oracle.dequantize_plain(qp, qs)[0, 0]
    kd = oracle.dequantize_plain(*oracle.quantize_plain(k))
    ref = np.maximum(kd @ qd, 0.0)
    assert np.array_equal(lg[0, :150], ref)


def test_brute_force_tiny_dense():
    ctx = [70, 33]
    lay, k, q, w, kv_p, kv_s, qp, qs = _decode_setup(32, ctx, 2)
    lg = oracle.decode_logits(qp, qs, w, kv_p, kv_s, lay.block_tables, np.array(ctx, np.int32))
    kd = oracle.dequantize_plain(*oracle.quantize_plain(k))
    qd = oracle.dequantize_plain(qp, qs)  # [B][H][128]
    start = 0
    for b, c in enumerate(ctx):
        s = np.einsum("hd,td->th", qd[b], kd[start:start + c])
        ref = np.maximum(s, 0.0) @ w[b].astype(np.float64)
        assert np.allclose(lg[b, :c], ref, rtol=1e-13, atol=1e-12)
        start += c


def test_exact_rational_tiny():
    ctx = [9]
    lay, k, q, w, kv_p, kv_s, qp, qs = _decode_setup(33, ctx, 3)
    lg = oracle.decode_logits(qp, qs, w, kv_p, kv_s, lay.block_tables, np.array(ctx, np.int32))
    kd = oracle.dequantize_plain(*oracle.quantize_plain(k))
    qd = oracle.dequantize_plain(qp, qs)[0]
    for t in range(9):
        total = Fraction(0)
        for h in range(3):
            s = sum(Fraction(float(qd[h, d])) * Fraction(float(kd[t, d])) for d in range(128))
            total += Fraction(float(w[0, h])) * max(s, Fraction(0))
        # the dot products are exact in fp64; only the final weighted head sum rounds
        assert abs(Fraction(float(lg[0, t])) - total) <= abs(total) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


def test_page_permutation_invariance_and_identity_table():
    ctx = [200]
    lay, k, q, w, kv_p, kv_s, qp, qs = _decode_setup(34, ctx, 4)
    ctx_a = np.array(ctx, np.int32)
    base = oracle.decode_logits(qp, qs, w, kv_p, kv_s, lay.block_tables, ctx_a)
    perm = synth.Rng(35).permutation(lay.num_pages)  # new page id of old page p is perm[p]
    kv_p2, kv_s2 = np.empty_like(kv_p), np.empty_like(kv_s)
    kv_p2[perm], kv_s2[perm] = kv_p, kv_s
    bt2 = lay.block_tables.copy()
    valid = bt2 >= 0
    bt2[valid] = perm[bt2[valid]]
    moved = oracle.decode_logits(qp, qs, w, kv_p2, kv_s2, bt2, ctx_a)
    assert np.array_equal(base, moved)
    # identity table over a flat pool: token t at slot t
    kv_p3, kv_s3 = _pool(4)
    assert oracle.quant_and_cache(k, np.arange(200, dtype=np.int32), kv_p3, kv_s3) == 200
    flat = oracle.decode_logits(qp, qs, w, kv_p3, kv_s3, np.arange(4, dtype=np.int32)[None], ctx_a)
    assert np.array_equal(base, flat)


def test_topk_against_library_sort():
    rng = synth.Rng(36)
    for n, k in [(1000, 64), (64, 64), (50, 64), (4097, 2048), (0, 16)]:
        for ties in (False, True):
            v = rng.normal(n)
            if ties:
                v = np.round(v * 4) / 4
            idx, val = oracle.select_topk(v, n, k)
            order = np.lexsort((np.arange(n), -v))[:min(k, n)]
            assert np.array_equal(idx[:len(order)], order)
            assert np.array_equal(val[:len(order)], v[order])
            assert np.all(idx[len(order):] == -1) and np.all(np.isneginf(val[len(order):]))


def test_padding_row_reads_no_key():
    # Two requests; the last one carries two padding rows with row_end 0. Key 0 of each
    # request and every unwritten row of the pool hold the NaN scale sentinel (0xFF).
    rng = synth.Rng(37)
    L = [40, 30]
    lay = synth.paged_layout(rng.fork(1), L)
    k = synth.qk_bf16(rng.fork(2), (sum(L),))
    kv_p, kv_s = _pool(lay.num_pages)
    slots = np.concatenate([lay.slots(0, 0, 40), lay.slots(1, 0, 30)])
    keep = np.ones(len(slots), bool)
    keep[[0, 40]] = False  # key 0 of both requests stays a NaN sentinel
    assert oracle.quant_and_cache(k[keep], slots[keep], kv_p, kv_s) == keep.sum()
    R = 6
    q = synth.qk_bf16(rng.fork(3), (R, 8))
    w = synth.head_weights(rng.fork(4), R, 8)
    qp, qs = oracle.quantize_plain(q)
    cu = np.array([0, 2, 6], np.int32)
    row_ends = np.array([40, 39, 30, 29, 0, 0], np.int32)
    idx, val, lg = oracle.prefill_topk(qp, qs, w, kv_p, kv_s, lay.block_tables, cu, row_ends, 16)
    assert np.all(idx[4:] == -1) and np.all(np.isneginf(val[4:]))
    # real rows read key 0 and are NaN there, which shows the sentinel is live
    assert np.isnan(lg[0, 0]) and np.isnan(lg[2, 0])
    # a row whose range starts past key 0 would be finite: check the finite part of row 0
    assert np.all(np.isfinite(lg[0, 1:40]))


def test_prefill_matches_decode_per_row():
    # A prefill row with row_end p+1 scores exactly what a decode row with ctx p+1 scores.
    rng = synth.Rng(38)
    L = [130]
    lay = synth.paged_layout(rng.fork(1), L)
    k = synth.qk_bf16(rng.fork(2), (130,))
    kv_p, kv_s = _pool(lay.num_pages)
    oracle.quant_and_cache(k, lay.slots(0, 0, 130), kv_p, kv_s)
    R = 5
    q = synth.qk_bf16(rng.fork(3), (R, 16))
    w = synth.head_weights(rng.fork(4), R, 16)
    qp, qs = oracle.quantize_plain(q)
    row_ends = np.array([1, 64, 65, 128, 130], np.int32)
    pl = oracle.prefill_logits(qp, qs, w, kv_p, kv_s, lay.block_tables, np.array([0, R], np.int32), row_ends)
    bt = np.repeat(lay.block_tables, R, axis=0)
    dl = oracle.decode_logits(qp, qs, w, kv_p, kv_s, bt, row_ends)
    for r in range(R):
        assert np.array_equal(pl[r, :row_ends[r]], dl[r, :row_ends[r]])
