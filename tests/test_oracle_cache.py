"""Pins for the oracle's paged index cache (CPU only).

Fixed by the pages: the scale plane stores a page's row axis as a 16x4 transpose
while the packed plane keeps it flat ("Score a DSA sparse indexer in FP4", review
finding 2 and the sub-commit on the index scale plane's row order), and the writer
skips negative slots (sub-commit "Schedule, refuse and document ...", second
instance of uninitialised reads). The byte offsets below are written from the
layout's definition, not read from the oracle.
"""
import numpy as np

import oracle
import synth

PAGE, G = 64, 4


def test_scale_slot_is_the_16x4_transpose():
    # View a page's 64 rows as a 4 x 16 matrix [row // 16][row % 16]; the scale plane stores
    # its transpose [row % 16][row // 16] flattened, so slot s holds the row at transposed[s].
    transposed = np.arange(64).reshape(4, 16).T.reshape(-1)
    for s in range(64):
        assert oracle.scale_slot(int(transposed[s])) == s
    slots = [oracle.scale_slot(r) for r in range(64)]
    assert sorted(slots) == list(range(64))  # a bijection on 0..63


def _pool(num_pages, packed_fill=0x77, scale_fill=0xFF):
    return (np.full((num_pages, G, PAGE, 16), packed_fill, np.uint8),
            np.full((num_pages, G, PAGE), scale_fill, np.uint8))


def test_writer_byte_offsets():
    rng = synth.Rng(21)
    k = synth.qk_bf16(rng, (3,))
    packed_plain, scales_plain = oracle.quantize_plain(k)
    kv_p, kv_s = _pool(5)
    slots = np.array([2 * 64 + 17, 4 * 64 + 63, 0], np.int32)
    assert oracle.quant_and_cache(k, slots, kv_p, kv_s) == 3
    flat_p, flat_s = kv_p.reshape(-1), kv_s.reshape(-1)
    for i, slot in enumerate(slots):
        page, row = divmod(int(slot), 64)
        for g in range(G):
            off = page * 4096 + g * 1024 + row * 16
            assert np.array_equal(flat_p[off:off + 16], packed_plain[i, 16 * g:16 * g + 16])
            soff = page * 256 + g * 64 + (row % 16) * 4 + row // 16
            assert flat_s[soff] == scales_plain[i, g]
    # every other byte keeps its sentinel
    written_p = np.zeros(flat_p.size, bool)
    written_s = np.zeros(flat_s.size, bool)
    for slot in slots:
        page, row = divmod(int(slot), 64)
        for g in range(G):
            written_p[page * 4096 + g * 1024 + row * 16:page * 4096 + g * 1024 + row * 16 + 16] = True
            written_s[page * 256 + g * 64 + (row % 16) * 4 + row // 16] = True
    assert np.all(flat_p[~written_p] == 0x77) and np.all(flat_s[~written_s] == 0xFF)


def test_writer_skips_negative_slots_and_flags_out_of_pool():
    rng = synth.Rng(22)
    k = synth.qk_bf16(rng, (4,))
    kv_p, kv_s = _pool(2)
    assert oracle.quant_and_cache(k, np.array([-1, -5, -1, -100], np.int32), kv_p, kv_s) == 0
    assert np.all(kv_p == 0x77) and np.all(kv_s == 0xFF)
    assert oracle.quant_and_cache(k, np.array([0, 128, 1, -1], np.int32), kv_p, kv_s) == -1


def test_write_read_round_trip():
    rng = synth.Rng(23)
    n = 300
    k = synth.qk_bf16(rng, (n,))
    lay = synth.paged_layout(rng.fork(1), [n])
    slots = lay.slots(0, 0, n)
    kv_p, kv_s = _pool(lay.num_pages)
    assert oracle.quant_and_cache(k, slots, kv_p, kv_s) == n
    ref = oracle.dequantize_plain(*oracle.quantize_plain(k))
    for t in range(n):
        page, row = divmod(int(slots[t]), 64)
        assert np.array_equal(oracle.read_key(kv_p, kv_s, page, row), ref[t])


def test_bytes_per_key_against_pool_pricing():
    # "Score a DSA sparse indexer in FP4", Performance: the index region prices a block
    # 102,144 B lower across 21 indexer layers, and the FP4/FP8 byte ratio is 0.47.
    path = __file__.replace("test_oracle_cache.py", "golden/pool_pricing.txt")
    fix = dict(ln.strip().split("=", 1) for ln in open(path) if ln.strip() and not ln.startswith("#"))
    block, layers, saving = int(fix["block_size"]), int(fix["indexer_layers"]), int(fix["block_saving_bytes"])
    kv_p, kv_s = _pool(1)
    fp4_per_key = (kv_p.nbytes + kv_s.nbytes) // block
    assert fp4_per_key == 68
    fp8_per_key = fp4_per_key + saving // (layers * block)
    assert saving % (layers * block) == 0
    assert round(fp4_per_key / fp8_per_key, 2) == float(fix["byte_ratio"])
