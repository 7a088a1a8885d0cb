"""The seeded input recipes: shapes, counts and determinism (no GPU)."""
import numpy as np
import torch

import workloads as W


def test_counts_are_multiples_of_256_and_offsets_cumulative():
    for name, fn in W.NAMED.items():
        w = fn()
        c = np.asarray(w.counts)
        assert c.shape == (w.num_experts,)
        assert np.all(c % (8 if w.unaligned else 256) == 0) and np.all(c >= 0), name
        assert int(w.offsets[-1]) == w.tokens_sum
        assert np.all(np.diff(np.concatenate([[0], w.offsets])) == c)


def test_tiny_counts():
    assert W.tiny().offsets.tolist() == [256, 768, 768, 1536]


def test_zipf_split():
    w = W.skewed()
    c = np.asarray(w.counts)
    assert w.tokens_sum == 262144
    assert int((c == 0).sum()) == 20
    assert int(c.max()) == 87296
    assert int(((c > 0) & (c <= 512)).sum()) + int((c == 0).sum()) == 85


def test_wide_has_two_zero_experts_and_accumulates():
    w = W.wide()
    assert int((np.asarray(w.counts) == 0).sum()) == 2
    assert w.accumulate and w.out_dtype == "bf16"


def test_round_to_256_is_nearest():
    assert W.round_to_256(np.array([127.9, 128.0, 383.9, 384.0, 0.0])).tolist() == [0, 256, 256, 512, 0]


def test_inputs_deterministic_and_shaped():
    w = W.custom(3, 128, 256, [256, 0, 512], seed=9, accumulate=True, out_dtype="bf16")
    x1 = W.make_inputs(w)
    x2 = W.make_inputs(w)
    assert torch.equal(x1.a.view(torch.int16), x2.a.view(torch.int16))
    assert x1.a.shape == (128, 768) and x1.b.shape == (768, 256)
    assert x1.c.shape == (3, 128, 256) and x1.c.dtype == torch.bfloat16
    assert x1.offsets.dtype == torch.int32


def test_ragged_packing_layout():
    counts = [256, 0, 512]
    a = torch.arange(4 * 768, dtype=torch.float32).reshape(4, 768).to(torch.bfloat16)
    flat = W.pack_ragged_a(a, np.array(counts))
    # expert 2 starts at element begin*hidden = 256*4 and has leading dimension 512
    blk = flat[256 * 4: 256 * 4 + 4 * 512].reshape(4, 512)
    assert torch.equal(blk, a[:, 256:768])


def test_fp8_inputs_have_scales():
    w = W.custom(2, 128, 256, [256, 256], seed=3, fp8=True, out_dtype="bf16")
    x = W.make_inputs(w)
    assert x.a.dtype == torch.float8_e4m3fn and x.b.dtype == torch.float8_e4m3fn
    assert x.sfa.shape == (4, 128) and x.sfb.shape == (4, 256)
    assert x.sfa.dtype == torch.float32


def test_fp4_quantiser_follows_the_rounding_rule():
    """The chunked torch quantiser rounds exactly like the plain per-element rule (nearest e2m1
    value, ties to the even code), including every midpoint."""
    import numpy as np
    import torch
    g = torch.Generator().manual_seed(5)
    x = torch.randn(48, 512, generator=g) * 3
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    x[0:2, :32] = 0.0
    x[0, :8], x[1, :8] = mids, -mids              # blocks with amax 6: scale 1, exact midpoints
    q, _ = W.quantize_e2m1_ue8m0_32(x, 1)
    xt = x.double().numpy().reshape(48, 16, 32)
    v = np.abs(xt).max(2) / 6.0
    fr, ex = np.frexp(v)
    k = np.where(v == 0, 0, np.where(fr == 0.5, ex - 1, ex))
    codes = W.e2m1_codes(xt / np.ldexp(1.0, k)[..., None]).reshape(48, 512)
    ref = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(q.numpy(), ref)
    assert q.numpy()[0, :4].tolist() == [0x20, 0x42, 0x64, 0x76]
    assert q.numpy()[1, :4].tolist() == [0xA0, 0xCA, 0xEC, 0xFE]


def test_unaligned_counts_are_multiples_of_8_not_all_of_256():
    c = np.asarray(W.unaligned().counts)
    assert np.all(c % 8 == 0) and np.any(c % 256 != 0) and np.any(c % 64 != 0)
