"""The seeded input generator and the I/O rounding, against their published definitions.

SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): the stateful
generator seeded with 0 starts 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4, ...; the counter form used here is the
same function of the counter.  bfloat16 keeps the top 16 bits of an fp32 value, rounding to nearest, ties to even."""
import numpy as np
import torch

from linear_attention_recurrence_delta_gb300 import inputs as I

SPLITMIX64_SEED0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC,
                    0x1B39896A51A8749B]


def test_splitmix64_reference_outputs():
    with np.errstate(over="ignore"):
        x = I._mix(np.arange(1, 6, dtype=np.uint64) * I._GOLDEN)
    assert [int(v) for v in x] == SPLITMIX64_SEED0


def test_uniform_and_normal():
    u = I.uniform(3, 1, 200000)
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.005
    z = I.normal(3, 2, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1.0) < 0.01
    # same (seed, stream) -> same values; another stream -> independent values
    np.testing.assert_array_equal(I.normal(3, 2, 1000), z[:1000])
    assert abs(np.corrcoef(I.normal(3, 1, 20000), I.normal(3, 2, 20000))[0, 1]) < 0.03


def test_streams_do_not_move_each_other():
    """The same workload always draws the same values; each tensor has its own stream, so a longer sequence
    leaves A_log as it was and (one batch row, [B, T, H, d] order) only appends tokens to v and g."""
    kw = dict(mode="delta", dtype="bf16", B=1, H=2, dk=8, dv=8, seed=4)
    a = I.make_inputs(I.custom(T=16, **kw))
    b = I.make_inputs(I.custom(T=16, **kw))
    for k in ("v", "b", "c", "g", "beta", "A_log"):
        np.testing.assert_array_equal(a[k], b[k])
    longer = I.make_inputs(I.custom(T=32, **kw))
    np.testing.assert_array_equal(a["A_log"], longer["A_log"])
    np.testing.assert_array_equal(a["v"], longer["v"][:, :16])
    np.testing.assert_array_equal(a["g"], longer["g"][:, :16])


def test_round_bf16_ties_to_even():
    one = 1.0
    assert I.round_bf16(np.array([one + 2.0 ** -8]))[0] == one                        # halfway, even below
    assert I.round_bf16(np.array([one + 3 * 2.0 ** -8]))[0] == one + 2.0 ** -6       # halfway, even above
    assert I.round_bf16(np.array([one + 2.0 ** -8 + 2.0 ** -30]))[0] == one + 2.0 ** -7
    assert I.round_bf16(np.array([-(one + 2.0 ** -8)]))[0] == -one
    exact = np.array([0.0, 1.0, -2.5, 3.0 * 2.0 ** -20, 65280.0])
    np.testing.assert_array_equal(I.round_bf16(exact), exact)


def test_round_bf16_matches_torch_on_fp32_values():
    x = (I.normal(5, 1, 200000) * np.exp(I.normal(5, 2, 200000) * 4)).astype(np.float32).astype(np.float64)
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(I.round_bf16(x), t)
