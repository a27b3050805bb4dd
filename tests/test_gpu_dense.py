"""A contiguous (non-paged) cache read through an identity block table.

"Three Attention Kernels" benchmarks split-KV decoding on dense K/V
(B 4, H 16, D 64, one query, fp16) and checks it against PyTorch's
scaled_dot_product_attention before timing ("Benchmark method").  Here the
same shapes go through pa_decode and pa_decode_splitkv + pa_merge with 1 to
128 splits and are compared with the fp64 oracle and with SDPA on the GPU.
"""

import pytest
import torch

import workloads
from helpers import assert_attn_close, oracle_seq

pytestmark = pytest.mark.gpu


def _read(lib, g, splits):
    out = torch.empty_like(g.q)
    if splits == 1:
        lib.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale)
        return out
    pps = max(1, g.max_blocks // splits)  # a split is at least one 16-token page
    s = lib.pa_num_splits(g.max_blocks, pps)
    po = torch.empty((g.num_seqs, g.num_q_heads, s, g.head_dim), device="cuda")
    pl = torch.empty((g.num_seqs, g.num_q_heads, s), device="cuda")
    lib.pa_decode_splitkv(po, pl, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale, pps)
    lib.pa_merge(out, po, pl)
    return out


def _sdpa(g, n):
    b, h, d = g.q.shape
    k = g.k_pool.reshape(b, n, h, d).transpose(1, 2)
    v = g.v_pool.reshape(b, n, h, d).transpose(1, 2)
    return torch.nn.functional.scaled_dot_product_attention(g.q.unsqueeze(2), k, v,
                                                            scale=g.scale).squeeze(2)


@pytest.mark.parametrize("n", [1024, 4096, 16384])
@pytest.mark.parametrize("splits", [1, 8, 32, 128])
def test_dense_matches_oracle_and_sdpa(lib, n, splits):
    g = workloads.dense(n, device="cuda")
    out = _read(lib, g, splits)
    ref_sdpa = _sdpa(g, n).double().cpu().numpy()
    assert_attn_close(out, ref_sdpa, g.dtype, "vs SDPA")
    for b in (0, 3):
        assert_attn_close(out[b], oracle_seq(g, b), g.dtype, f"seq {b} vs oracle")
