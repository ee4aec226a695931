"""The input generator: published test vectors of its RNGs and the properties of
the inputs it builds (CPU only)."""
import numpy as np
import pytest

import synth


def test_pcg32_reference_output():
    # pcg32 demo stream (initstate 42, initseq 54): first six outputs
    got = synth.pcg32_raw(6, 42, 54).tolist()
    assert got == [0xA15C02B7, 0x7B47F409, 0xBA1D3330, 0x83D2F293, 0xBFA4784B, 0xCBED606E]


def test_splitmix64_reference_output():
    assert synth.splitmix64_raw(3, 0).tolist() == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                                  0x06C45D188009454F]
    assert synth.splitmix64_raw(2, 1234567).tolist() == [6457827717110365317, 3203168211198807973]


def test_fp16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.uniform(0.01, 0.05, 20000), rng.uniform(-3, 3, 2000),
                           rng.uniform(0, 1e-5, 2000)])
    # exact midpoints between fp16 neighbours: ties to even
    base = np.arange(1024, 1100, dtype=np.float64)
    vals = np.concatenate([vals, (base + 0.5) * 2.0 ** -10 * 0.03125])
    for v in vals:
        assert synth.lib().synth_fp16_rne(float(v)) == int(np.float16(v).view(np.uint16)), v


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(1).standard_normal(5000).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([synth.lib().synth_bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_store_layout_and_scales():
    H, F = 256, 512
    st = synth.store(1, 2, H, F, seed=0)
    assert st.size == 2 * synth.expert_bytes(H, F) == 2 * 221_184
    blocks = st.reshape(-1, 18)
    d = blocks[:, 0:2].copy().view(np.float16)[:, 0].astype(np.float64)
    assert d.min() >= 0.0099 and d.max() <= 0.0501
    nib = np.concatenate([blocks[:, 2:] & 0xF, blocks[:, 2:] >> 4]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * counts.mean()
    # expert blocks are independent streams and reproducible
    assert np.array_equal(st[: synth.expert_bytes(H, F)], synth.expert_block(0, 0, H, F, 0))
    assert not np.array_equal(st[: 1000], st[synth.expert_bytes(H, F): synth.expert_bytes(H, F) + 1000])


def test_store_thread_count_does_not_change_bytes():
    a = synth.store(2, 3, 256, 512, seed=3, threads=1)
    b = synth.store(2, 3, 256, 512, seed=3, threads=4)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("E,k,s,p", [(128, 8, 1.1, 0.39), (256, 8, 1.0, 0.30), (128, 8, 0.0, 0.0),
                                     (8, 2, 0.0, 0.5)])
def test_trace_and_logits(E, k, s, p):
    n = 300
    picks = synth.trace(n, E, k, s, p, seed=0, layer=1, stream=2)
    assert picks.min() >= 0 and picks.max() < E
    for t in range(n):
        assert len(set(picks[t].tolist())) == k
    lg = synth.logits_from_picks(picks, E, seed=0, layer=1, stream=2)
    for t in range(n):
        top = set(np.argsort(-lg[t], kind="stable")[:k].tolist())
        assert top == set(picks[t].tolist())
        assert len(set(lg[t][picks[t]].tolist())) == k   # no exact ties among the picked
    if p > 0:
        ov = np.mean([len(set(picks[t]) & set(picks[t - 1])) / k for t in range(1, n)])
        assert ov >= p - 0.05


def test_zipf_skew():
    E = 128
    picks = synth.trace(2000, E, 8, 1.1, 0.0, seed=0, layer=0, stream=0)
    perm = synth.permutation(E, 0, 0)
    counts = np.bincount(picks.ravel(), minlength=E)
    # the rank-1 expert is the most used, rank E among the least
    assert counts[perm[0]] == counts.max()
    assert counts[perm[-1]] < counts[perm[0]] / 10
