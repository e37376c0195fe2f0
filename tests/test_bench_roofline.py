"""The roofline numerators bench.py reports, derived independently of its own
formulas: the packed bytes a decode step reads and a prefill write stores come
from the oracle's cache layout (a page's bytes over its token slots, K and V of
every kv head), the token counts from the workloads' seeded lengths; the
prefill-attention flops from the closed form of the causal sum.  No GPU: the
workload objects are stood in for by their parameters."""
from types import SimpleNamespace

import numpy as np

import bench
from oracle import kvq3_oracle as O


def _bytes_per_token(w):
    """Packed bytes of one token (K and V of every kv head) in the oracle's layout."""
    lay = O.Layout(w.d, w.num_kv_heads, w.block, w.scale, w.page_size, 1, 1, 1, w.bits)
    assert lay.page_bytes % w.page_size == 0
    return lay.page_bytes // w.page_size


def test_decode_bytes_match_the_oracle_layout():
    quoted = {"llama8b": 436_600_832, "long70b": 839_254_016, "ragged": 1_936_127_616}
    for name, want in quoted.items():
        w = bench.workload(name)
        lens = bench.workload_lens(w)
        packed = int(np.sum(lens, dtype=np.int64)) * _bytes_per_token(w)
        q_out = w.batch * w.num_q_heads * w.d * (2 + 4)          # fp16 queries in, fp32 outputs out
        got = bench.algorithmic_bytes(w, lens)
        assert got["decode"] == packed + q_out == want, name
        assert got["per_token_head"] * w.num_kv_heads == _bytes_per_token(w)


def test_prefill_write_bytes_match_the_oracle_layout():
    w = bench.workload("prefill")
    n_vec = w.seq_len * w.num_kv_heads * 2                        # K and V vectors
    want = n_vec * w.d * 2 + w.seq_len * _bytes_per_token(w)      # fp16 in, packed out
    assert bench.PrefillWorkload.bytes(SimpleNamespace(w=w)) == want == 671_088_640


def test_prefill_attention_flops_closed_form():
    # query i at pos0 + i attends to pos0 + i + 1 keys; QK^T and PV are
    # 2 d multiply-adds (4 d flops) per (query head, key)
    w = bench.workload("prefill_attn")
    n, pos0 = w.chunk, w.seq_len - w.chunk
    closed = 4 * w.d * w.num_q_heads * (n * pos0 + n * (n + 1) // 2)
    got = bench.PrefillAttnWorkload.flops(SimpleNamespace(w=w, pos0=pos0))
    assert got == closed == 1_065_168_666_624
