"""The seeded input generator: bf16 rounding, layout and poison placement."""
import numpy as np

from mla_latent_cache_gb300 import workloads as W


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 0.0, 3.0e38], dtype=np.float32)
    bits = W.f32_to_bf16_bits(x)
    # 1+2^-8 is a tie between 1.0 and 1+2^-7 -> even (1.0); 1+3*2^-8 ties -> 1+2^-6 (even mantissa)
    assert bits.tolist()[:6] == [0x3F80, 0x3F80, 0x3F82, 0x3F80, 0xC020, 0x0000]
    back = W.bf16_bits_to_f64(bits)
    assert back[0] == 1.0 and back[2] == 1.0 + 2**-6 and back[4] == -2.5
    assert np.all(np.abs(W.bf16_bits_to_f64(W.f32_to_bf16_bits(x[:5])) - x[:5]) <= np.abs(x[:5]) * 2**-8)


def test_workload_layout_and_poison():
    w = W.custom_workload(16, [70, 1, 128, 0], T=1, seed=3)
    assert w.block_table.shape == (4, 2)
    assert (w.block_table[1, 1:] == -1).all() and (w.block_table[3] == -1).all()
    pool = w.full_pool()
    used = set(w.pool_ids.tolist())
    for blk in range(w.num_blocks):
        if blk not in used:
            assert (pool[blk] == W.BF16_NAN).all()
    # sequence 0 has 70 rows: its second page holds 6 real rows then NaN
    p1 = pool[w.block_table[0, 1]]
    assert not (p1[:6] == W.BF16_NAN).any() and (p1[6:] == W.BF16_NAN).all()
    # compact view resolves the same rows
    cp, cbt = w.compact_view()
    for b in range(4):
        for pg in range((int(w.seq_lens[b]) + 63) // 64):
            assert np.array_equal(cp[cbt[b, pg]], pool[w.block_table[b, pg]])


def test_named_workloads_shapes_and_determinism():
    w1 = W.config_workload(1)
    assert (w1.H, w1.B, w1.T, w1.num_blocks) == (16, 1, 1, 8)
    assert sorted(w1.block_table[0].tolist()) == list(range(8))
    w1b = W.config_workload(1)
    assert np.array_equal(w1.pool_data, w1b.pool_data) and np.array_equal(w1.q_nope, w1b.q_nope)
    wu = W.bf16_bits_to_f64(w1.w_uk)
    assert abs(wu.std() - 1 / np.sqrt(512)) < 0.002
    assert abs(W.bf16_bits_to_f64(w1.q_nope).std() - 0.1) < 0.01
    w3 = W.config_workload(3)
    assert w3.B == 128 and w3.seq_lens.min() >= 256 and w3.seq_lens.max() <= 32768
    ids = w3.block_table[w3.block_table >= 0]
    assert len(np.unique(ids)) == len(ids)
    w5 = W.config_workload(5, T=64)
    assert (w5.seq_lens == 8192 + 64).all() and w5.causal and w5.T == 64
