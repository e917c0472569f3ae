"""The seeded input generator: its random stream, distributions, rounding and layouts (CPU)."""
import numpy as np
import pytest

import synth


def test_philox_published_known_answer():
    # Random123 known-answer vector for philox4x64-10 with zero counter and zero key.
    assert synth.philox4x64_10([0, 0, 0, 0], [0, 0]) == [
        0x16554D9ECA36314C, 0xDB20FE9D672D0FDC, 0xD7E772CEE186176B, 0x7E68B68AEC7BA23B]


@pytest.mark.parametrize("ctr,key", [(0, (0, 0)), (41, (7, 9)), (2 ** 40 + 5, (123456789, 2 ** 52 + 11))])
def test_philox_matches_numpy(ctr, key):
    # numpy's Philox bit generator is philox4x64-10; it advances the counter before each block.
    bg = np.random.Philox(counter=[ctr, 0, 0, 0], key=list(key))
    ref = [int(x) for x in bg.random_raw(4)]
    assert synth.philox4x64_10([ctr + 1, 0, 0, 0], list(key)) == ref


def test_normal_moments():
    z = synth.normal_f64(11, 1, 2, 3, 0, 1 << 22)
    assert abs(z.mean()) < 3e-3
    assert abs(z.std() - 1.0) < 3e-3
    # two-sided tail beyond 3 sigma: 0.27%
    assert abs((np.abs(z) > 3).mean() - 0.0027) < 3e-4


def test_random_access_equals_contiguous():
    wl = synth.WORKLOADS["llama7b_16l"]
    g = synth.grads_bf16(wl, 1, 1, 1000, 5000)
    idx = np.array([1000, 1001, 1002, 2345, 5999, 4444])
    assert np.array_equal(synth.grads_bf16_at(wl, 1, 1, idx), g[idx - 1000])
    # odd start: the pair split must not shift values
    assert np.array_equal(synth.grads_bf16(wl, 1, 1, 1001, 10), g[1:11])
    m = synth.master_f32(wl, 77, 100)
    assert np.array_equal(synth.master_f32_at(wl, np.arange(77, 177)), m)


def test_heavy_tail_fraction():
    wl = synth.WORKLOADS["llama7b_16l"]
    g = synth.grads_bf16(wl, 0, 0, 0, 1 << 21)
    x = (g.astype(np.uint32) << 16).view(np.float32)
    frac = (np.abs(x) > 6e-4).mean()   # > 6 sigma of the bulk: essentially only outliers
    assert abs(frac - 0.01 * 0.95) < 1.5e-3


def test_bf16_rounding_vs_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    # fp32-exact inputs, so the library's rounding (via fp32) is a single rounding too
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32).astype(np.float64)
    x = x[np.isfinite(x)]
    mine = np.array([synth.f64_to_bf16_bits(v) for v in x], dtype=np.uint16)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_rounding_ties_and_edges():
    one = 0x3F80
    assert synth.f64_to_bf16_bits(1.0 + 2 ** -8) == one              # tie -> even
    assert synth.f64_to_bf16_bits(1.0 + 3 * 2 ** -8) == one + 2      # tie -> even (up)
    assert synth.f64_to_bf16_bits(1.0 + 2 ** -8 + 2 ** -40) == one + 1   # just above the tie
    assert synth.f64_to_bf16_bits(-0.0) == 0x8000
    assert synth.f64_to_bf16_bits(float("inf")) == 0x7F80
    assert synth.f64_to_bf16_bits(3.5e38) == 0x7F80                  # beyond bf16 max
    assert synth.f64_to_bf16_bits(2 ** -133) == 0x0001               # smallest subnormal
    assert synth.f64_to_bf16_bits(2 ** -134) == 0x0000               # tie at half the smallest -> even (0)


def test_param_list_sizes():
    assert synth.numel(synth.gpt2_small_shapes()) == 123_568_896
    assert synth.numel(synth.gpt_1p3b_shapes()) == 1_311_082_496
    assert synth.numel(synth.llama7b_16l_shapes()) == 3_238_133_760
    offs = synth.flatten_offsets(synth.gpt2_small_shapes())
    assert offs[0] == 0 and offs[1] == 50257 * 768


def _check_layout(segs, psi, n):
    g = 0
    per_owner = {}
    for go, ln, o, lo in segs:
        assert go == g and ln >= 0 and 0 <= o < n and lo >= 0
        g += ln
        per_owner.setdefault(o, []).append((lo, ln))
    assert g == psi
    for o, rs in per_owner.items():
        rs.sort()
        cur = 0
        for lo, ln in rs:
            assert lo == cur
            cur += ln


@pytest.mark.parametrize("psi,n", [(0, 3), (7, 8), (1 << 20, 2), ((1 << 20) + 3, 8), (123_568_896, 8)])
def test_layouts_cover_space(psi, n):
    _check_layout(synth.layout_even(psi, n), psi, n)
    _check_layout(synth.layout_ragged(psi, n, 3), psi, n)
    if psi > 0:
        _check_layout(synth.layout_random(psi, n, 9, 4), psi, n)
        _check_layout(synth.layout_buckets(psi, n, max(1, psi // 5), 3), psi, n)


def test_bucket_layout_is_misaligned():
    wl = synth.WORKLOADS["gpt_1p3b"]
    segs = synth.layout_of(wl)
    _check_layout(segs, wl.psi, wl.n)
    assert len(segs) == 53 * 8
    interior = [go for go, ln, o, lo in segs if o != 0]
    assert all(go % 4 != 0 and go % 8 != 0 for go in interior)
    # per bucket the last shard is 3 shorter than the middle ones
    assert segs[7][1] == segs[6][1] - 3 and segs[0][1] == segs[1][1] + 3
