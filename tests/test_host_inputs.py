"""Host-side logic on CPU: the seeded workload generators' structure (paged layouts, the flat
staged layout, verify rows of speculative decoding) and the benchmark's bookkeeping that does not
need a GPU (algorithmic bytes, the profile's code hash)."""
import numpy as np

import bench
import synth


def test_random_layout_partitions_pool():
    lay = synth.paged_layout(synth.Rng(3), [300, 64, 1, 0, 129])
    used = np.concatenate(lay.seq_pages)
    assert used.size == len(set(used.tolist()))              # no page shared between sequences
    assert np.all(used >= 0) and np.all(used < lay.num_pages)
    assert [p.size for p in lay.seq_pages] == [5, 1, 1, 0, 3]
    assert lay.num_pages >= 10 + 1                           # 12.5 % spare, at least one page


def test_contiguous_layout_is_identity_per_sequence():
    lay = synth.paged_layout(synth.Rng(3), [300, 64, 129], spare=0.0, contiguous=True)
    assert lay.num_pages == 5 + 1 + 3
    assert np.array_equal(lay.block_tables[0, :5], np.arange(5))
    assert np.array_equal(lay.block_tables[1, :1], [5])
    assert np.array_equal(lay.block_tables[2, :3], [6, 7, 8])
    assert np.all(lay.block_tables[1, 1:] == -1)


def test_flat_prefill_workload_shape():
    case = synth.prefill_flat_config()
    assert case.prompt_lens.tolist() == [16384]
    assert np.array_equal(case.layout.block_tables[0], np.arange(256))
    ends = np.concatenate([st.row_ends[:st.real_rows] for st in case.steps])
    assert np.array_equal(ends, np.arange(1, 16385))         # causal: row at position p sees p + 1 keys
    assert all(st.rows % 8 == 0 and st.rows <= 512 for st in case.steps)


def test_verify_rows_see_a_causal_suffix():
    case = synth.mtp_case("t", 1, [300, 3, 70], 16, 64, 3)
    assert case.q_bf16.shape == (9, 16, 128) and case.w.shape == (9, 16)
    assert case.row_ends().tolist() == [298, 299, 300, 1, 2, 3, 68, 69, 70]
    assert case.cu_seqlens().tolist() == [0, 3, 6, 9]
    big = synth.mtp_config()
    assert big.next_n == 2 and big.batch == 16 and int(big.row_ends().max()) == 131072


def test_decode_alg_bytes_counts_keys_pages_queries_outputs():
    # one sequence of 65 keys: 2 pages; 4 heads; top-8
    assert bench.decode_alg_bytes([65], 4, 8) == 68 * 65 + 4 * 2 + 4 * 72 + 8 * 8
    assert bench.decode_alg_bytes([0, 64], 1, 1) == (72 + 8) + (68 * 64 + 4 + 72 + 8)


def test_code_hash_ignores_comments_not_code():
    a = 'int f() { return 1; } // one\n/* block\n comment */ const char* s = "x // y";'
    b = 'int f() {\n  return 1;   // a different comment\n}\n const char* s = "x // y";'
    c = 'int f() { return 2; } const char* s = "x // y";'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert '"x // y"' in bench._code_only(a)               # string literals are code
