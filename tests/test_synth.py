"""The seeded input generators: determinism, ranges and the stated statistics."""
import numpy as np
import torch

import synth


def test_mul32_exact():
    rnd = np.random.default_rng(0)
    a = rnd.integers(0, 2 ** 32, size=2000, dtype=np.int64)
    for c in (0x85EBCA6B, 0xC2B2AE35, 1, 0xFFFFFFFF):
        got = synth._mul32(torch.from_numpy(a), c).numpy()
        ref = np.array([(int(x) * c) % 2 ** 32 for x in a])
        assert np.array_equal(got, ref)


def test_hash_and_normals():
    c = torch.arange(0, 1000, dtype=torch.int64)
    h1 = synth.hash32(0, 5, c)
    assert torch.equal(h1, synth.hash32(0, 5, c)) and not torch.equal(h1, synth.hash32(1, 5, c))
    assert int(h1.min()) >= 0 and int(h1.max()) < 2 ** 32
    z = synth.normal(3, 7, 0, 400_000)
    assert abs(float(z.mean())) < 0.01 and abs(float(z.std()) - 1) < 0.01
    # chunked generation gives the same tensor as one piece
    w1 = synth.make_weight(synth.TINY, "l0.wq", 0, chunk=1000)
    w2 = synth.make_weight(synth.TINY, "l0.wq", 0)
    assert torch.equal(w1, w2) and abs(float(w2.std()) - 0.02) < 0.001


def test_prompts():
    p = synth.uniform_prompt(512, 32, 1)
    assert p.dtype == np.int32 and len(p) == 32 and p.min() >= 0 and p.max() < 512
    m1 = synth.markov_zipf_prompt(32000, 512, 2)
    assert np.array_equal(m1, synth.markov_zipf_prompt(32000, 512, 2))
    assert m1.min() >= 0 and m1.max() < 32000
    c = synth.code_like_prompt(32000, 2048, 4)
    assert len(c) == 2048 and 0.15 < synth.code_like_prompt.last_copied_fraction < 0.45


def test_markov_rank_law():
    """Next-token ranks follow the truncated Zipf law: rank 1 has mass cdf[0]."""
    mc = synth.MarkovZipf(512, 9)
    n = 20000
    r1 = sum(int(np.searchsorted(mc.cdf, mc._u(), side="left")) == 0 for _ in range(n))
    assert abs(r1 / n - mc.cdf[0]) < 4 * np.sqrt(mc.cdf[0] * (1 - mc.cdf[0]) / n)


def test_wo_scale_scales_only_the_attention_output_exactly():
    """A power-of-two scale changes the wo tensors by exactly that factor
    (bf16 and fp32 storage) and leaves every other tensor alone; other
    scales are refused."""
    import dataclasses
    import pytest
    import torch
    for cfg in (synth.TINY, dataclasses.replace(synth.TINY, dtype="bf16")):
        a = synth.llama_weights(cfg, 3)
        b = synth.llama_weights(cfg, 3, wo_scale=2.0 ** -10)
        for n in a:
            if n.endswith(".wo"):
                assert torch.equal(b[n].float(), a[n].float() * 2.0 ** -10)
            else:
                assert torch.equal(a[n], b[n])
    with pytest.raises(AssertionError):
        synth.llama_weights(synth.TINY, 0, wo_scale=0.001)
