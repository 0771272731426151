"""Host-side arithmetic of the benchmark, on the CPU: the counts its JSON line
reports are checked against closed forms and against brute-force enumeration."""

import numpy as np

import bench
import workloads


def _brute_pairs(b, window=0):
    """Enumerate every (query, key) pair the attention scores."""
    total = 0
    qsl = b.query_start_loc
    for r, n in enumerate(b.seq_lens):
        n, q = int(n), int(qsl[r + 1] - qsl[r])
        for j in range(q):
            p = n - q + j
            for t in range(n):
                if b.causal and t > p:
                    continue
                if window and t < p - window + 1:
                    continue
                total += 1
    return total


def test_decode_pairs_are_the_context_tokens():
    b = workloads.tiny()
    assert bench.qk_pairs(b) == int(b.seq_lens.sum()) == 17 + 64 + 129 + 200
    # a window of 32 keeps min(len, 32) keys per sequence
    assert bench.qk_pairs(b, 32) == 17 + 32 + 32 + 32


def test_chunk_pairs_closed_form_and_brute_force():
    b = workloads.build("qk", 3, [70, 9, 33], [20, 1, 33], 8, 2, 64, 16, "bf16")
    # a causal chunk of q tokens ending at n scores q (n - q + 1) + q (q - 1) / 2 pairs
    want = sum(q * (n - q + 1) + q * (q - 1) // 2 for n, q in ((70, 20), (9, 1), (33, 33)))
    assert bench.qk_pairs(b) == want == _brute_pairs(b)
    for w in (1, 5, 40):
        assert bench.qk_pairs(b, w) == _brute_pairs(b, w)


def test_non_causal_rows_score_the_whole_context():
    b = workloads.build("qk_nc", 4, [50, 12], [10, 12], 8, 2, 64, 16, "bf16", causal=False)
    assert bench.qk_pairs(b) == 10 * 50 + 12 * 12 == _brute_pairs(b)


def test_empty_requests_score_nothing():
    b = workloads.build("qk_empty", 5, [10, 30], [0, 2], 8, 2, 64, 16, "bf16")
    assert bench.qk_pairs(b) == 29 + 30 == _brute_pairs(b)
    assert np.diff(b.query_start_loc).tolist() == [0, 2]


def test_byte_counts_of_the_agentic_forks():
    """The headline's byte basis, from closed forms.  Forks share floor(0.96 * blocks)
    whole blocks with their parent: the unique K/V tokens are each parent's whole context
    plus each fork's private remainder; the shared-prefix split (each family's shared
    prefix once, every sequence's private rest) covers exactly those bytes; the logical
    bytes are every sequence's whole context."""
    b = workloads.agentic(seed=2, host_cache=False, scale_lengths=1 / 300.0)
    bs = b.block_size
    kv_tok = 2 * b.num_kv_heads * b.head_size * workloads.ELEM_BYTES[b.kv_dtype]
    unique = 0
    for fam in b.families:
        L = int(b.seq_lens[fam[0]])
        if len(fam) == 1:
            unique += L
            continue
        nshare = int(np.floor(0.96 * -(-L // bs)))
        unique += L + (len(fam) - 1) * (L - nshare * bs)
    assert bench.unique_kv_tokens(b) == unique
    split = bench.shared_split_bytes(b, bench.prefix_groups(b))
    assert split["shared"] + split["private"] == unique * kv_tok
    nb = bench.algorithmic_bytes(b)
    assert nb["unique_kv"] == unique * kv_tok
    assert nb["logical_kv"] == int(b.seq_lens.sum()) * kv_tok
    q_out = 2 * b.num_seqs * b.num_q_heads * b.head_size * workloads.ELEM_BYTES[b.q_dtype]
    tables = 4 * sum(-(-int(n) // bs) for n in b.seq_lens) + 4 * b.num_seqs
    assert nb["algorithmic"] == unique * kv_tok + q_out + tables
    assert nb["logical_total"] == int(b.seq_lens.sum()) * kv_tok + q_out + tables


def test_unique_bytes_without_sharing_are_the_logical_bytes():
    b = workloads.build("noshare", 6, [100, 17, 64], [1, 1, 1], 8, 2, 64, 16, "bf16", host_cache=False)
    nb = bench.algorithmic_bytes(b)
    assert nb["unique_kv"] == nb["logical_kv"] == (100 + 17 + 64) * 2 * 2 * 64 * 2
