"""Pins for the fp64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: a library
routine (torch's fp64 scaled_dot_product_attention / logsumexp), a closed form,
or an invariant of masked softmax attention.  The definition being pinned is
the one in ``oracle.attention`` (Tessera abstract: only the interactions the
logical block mask selects are computed, and they are preserved exactly).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as OA
from block_sparse_attention_plan_gb300 import workloads as W


def _token_mask(mask, bq, bk):
    """Token-level boolean mask by library repeat (independent of the oracle)."""
    return (mask != 0).repeat_interleave(bq, dim=2).repeat_interleave(bk, dim=3)


def _sdpa(q, k, v, mask, bq, bk, scale=None):
    g = q.shape[1] // k.shape[1]
    k64 = k.double().repeat_interleave(g, dim=1)
    v64 = v.double().repeat_interleave(g, dim=1)
    tm = _token_mask(mask, bq, bk)
    o = F.scaled_dot_product_attention(q.double(), k64, v64, attn_mask=tm, scale=scale)
    s = (q.double() @ k64.transpose(-1, -2)) * (scale if scale is not None else 1 / math.sqrt(q.shape[-1]))
    s = s.masked_fill(~tm, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    nonempty = tm.any(dim=-1)
    return o.numpy(), lse.numpy(), nonempty.numpy()


def _problem(seed, B, Hq, Hkv, Nq, Nk, d, bq, bk, p):
    return W.random_problem(seed, B, Hq, Hkv, Nq, Nk, d, bq, bk, p)


@pytest.mark.parametrize("bq,bk,d", [(64, 32, 64), (32, 128, 32), (128, 64, 16)])
def test_matches_sdpa_with_boolean_mask_gqa(bq, bk, d):
    w = _problem(1, 2, 4, 2, 256, 384, d, bq, bk, 0.35)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk)
    Os, Ls, ne = _sdpa(w.q, w.k, w.v, w.mask, bq, bk)
    assert ne.any()
    np.testing.assert_allclose(O[ne], Os[ne], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L[ne], Ls[ne], rtol=1e-12, atol=1e-12)
    assert np.all(O[~ne] == 0.0) and np.all(np.isneginf(L[~ne]))


def test_dense_form_matches_sdpa_and_gather_form():
    w = _problem(2, 1, 2, 1, 128, 192, 16, 32, 64, 0.4)
    Od, Ld = OA.dense_masked(w.q, w.k, w.v, w.mask, 32, 64)
    Og, Lg = OA.block_gather(w.q, w.k, w.v, w.mask, 32, 64)
    Os, Ls, ne = _sdpa(w.q, w.k, w.v, w.mask, 32, 64)
    np.testing.assert_allclose(Od[ne], Os[ne], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Od, Og, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(Ld), np.isneginf(Lg))
    np.testing.assert_allclose(Ld[ne], Lg[ne], rtol=1e-13)


def test_all_ones_mask_is_dense_sdpa():
    w = _problem(3, 1, 3, 3, 256, 256, 32, 64, 64, 1.1)
    assert bool((w.mask != 0).all())
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 64)
    o = F.scaled_dot_product_attention(w.q.double(), w.k.double(), w.v.double()).numpy()
    np.testing.assert_allclose(O, o, rtol=1e-10, atol=1e-12)
    s = (w.q.double() @ w.k.double().transpose(-1, -2)) / math.sqrt(32)
    np.testing.assert_allclose(L, torch.logsumexp(s, -1).numpy(), rtol=1e-12)


def test_empty_rows_give_zero_and_neg_inf():
    w = _problem(4, 1, 2, 2, 256, 256, 32, 64, 64, 0.5)
    w.mask[0, 1, 2, :] = 0
    w.mask[0, 0, :, :] = 0
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 64)
    assert np.all(O[0, 0] == 0) and np.all(np.isneginf(L[0, 0]))
    assert np.all(O[0, 1, 128:192] == 0) and np.all(np.isneginf(L[0, 1, 128:192]))
    assert np.all(np.signbit(O[0, 0]) == False)  # +0.0, not -0.0


def test_identical_keys_give_mean_of_selected_values():
    # All keys equal: every selected score is the same s = scale*<q, k>, so the
    # softmax is uniform over J: O = mean of the selected V rows, LSE = s + ln|J|.
    w = _problem(5, 1, 2, 2, 128, 256, 32, 32, 64, 0.5)
    kvec = torch.randn(32, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    k = kvec.expand(1, 2, 256, 32).contiguous()
    O, L = OA.block_gather(w.q, k, w.v, w.mask, 32, 64)
    q64, k64, v64 = w.q.double().numpy(), kvec.double().numpy(), w.v.double().numpy()
    m = w.mask.numpy()
    for h in range(2):
        for i in range(128):
            kbs = np.flatnonzero(m[0, h, i // 32])
            if kbs.size == 0:
                assert np.isneginf(L[0, h, i])
                continue
            keys = np.concatenate([np.arange(kb * 64, kb * 64 + 64) for kb in kbs])
            s = float(q64[0, h, i] @ k64) / math.sqrt(32)
            np.testing.assert_allclose(O[0, h, i], v64[0, h, keys].mean(axis=0), rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(L[0, h, i], s + math.log(keys.size), rtol=1e-12, atol=1e-12)


def test_single_selected_block_is_dense_attention_on_that_block():
    w = _problem(6, 1, 1, 1, 256, 512, 64, 128, 128, 0.0)
    w.mask.zero_()
    w.mask[0, 0, 0, 3] = 1
    w.mask[0, 0, 1, 0] = 1
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128)
    for qb, kb in [(0, 3), (1, 0)]:
        qs = w.q[:, :, qb * 128:(qb + 1) * 128].double()
        ks = w.k[:, :, kb * 128:(kb + 1) * 128].double()
        vs = w.v[:, :, kb * 128:(kb + 1) * 128].double()
        o = F.scaled_dot_product_attention(qs, ks, vs).numpy()
        np.testing.assert_allclose(O[:, :, qb * 128:(qb + 1) * 128], o, rtol=1e-10, atol=1e-12)


def test_softmax_normalisation_and_scale_override():
    w = _problem(7, 1, 2, 2, 128, 256, 64, 64, 64, 0.6)
    scale = 0.37
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 64, scale=scale)
    Os, Ls, ne = _sdpa(w.q, w.k, w.v, w.mask, 64, 64, scale=scale)
    np.testing.assert_allclose(O[ne], Os[ne], rtol=1e-10, atol=1e-12)
    # sum_j exp(s_j - LSE) = 1 over the selected keys
    s = (w.q.double() @ w.k.double().transpose(-1, -2)) * scale
    tm = _token_mask(w.mask, 64, 64)
    p = torch.exp(s - torch.from_numpy(L)[..., None]).masked_fill(~tm, 0.0).sum(-1).numpy()
    np.testing.assert_allclose(p[ne], 1.0, rtol=1e-12)


def test_affine_equivariance_in_v():
    w = _problem(8, 1, 2, 1, 128, 128, 32, 32, 32, 0.5)
    a, b = 2.5, -0.75
    O1, L1 = OA.block_gather(w.q, w.k, w.v, w.mask, 32, 32)
    v2 = w.v.double() * a + b
    O2, L2 = OA.block_gather(w.q, w.k, v2, w.mask, 32, 32)
    ne = np.isfinite(L1)
    np.testing.assert_allclose(O2[ne], a * O1[ne] + b, rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(L1, L2)


def test_sampled_rows_match_full_gather():
    w = W.make_workload("long_video_dit_small")
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128)
    samples = [(0, 0, 0), (0, 3, 10), (0, 2, 9), (0, 1, 4)]
    got = OA.sampled_qblocks(w.q, w.k, w.v, w.mask, 128, 128, samples)
    for (b, h, qb), (o, l) in got.items():
        np.testing.assert_array_equal(o, O[b, h, qb * 128:(qb + 1) * 128])
        np.testing.assert_array_equal(l, L[b, h, qb * 128:(qb + 1) * 128])
    # the all-padding block selects nothing: empty rows
    assert np.all(np.isneginf(L[0, :, 10 * 128:]))


# ---------------------------------------------------------------- element mask
def test_causal_equals_sdpa_is_causal():
    # Nq = Nk, all-ones block mask: the element mask is plain causal attention.
    w = _problem(41, 1, 2, 2, 128, 128, 32, 32, 32, 1.0)
    ones = torch.ones(1, 2, 4, 4, dtype=torch.uint8)
    O, L = OA.dense_masked(w.q, w.k, w.v, ones, 32, 32, causal=True)
    ref = F.scaled_dot_product_attention(w.q.double(), w.k.double(), w.v.double(), is_causal=True)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)


def test_causal_offset_equals_shifted_tril_mask():
    # Nq < Nk: queries are the last Nq positions, so query i sees keys j <= i + Nk - Nq;
    # the mask here is built with torch.tril's diagonal offset.
    w = _problem(42, 1, 2, 1, 64, 192, 32, 32, 32, 1.0)
    ones = torch.ones(1, 2, 2, 6, dtype=torch.uint8)
    O, L = OA.dense_masked(w.q, w.k, w.v, ones, 32, 32, causal=True)
    tm = torch.ones(64, 192, dtype=torch.bool).tril(diagonal=192 - 64)
    k64 = w.k.double().repeat_interleave(2, dim=1)
    v64 = w.v.double().repeat_interleave(2, dim=1)
    ref = F.scaled_dot_product_attention(w.q.double(), k64, v64, attn_mask=tm)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)
    s = (w.q.double() @ k64.transpose(-1, -2)) / math.sqrt(32)
    lse = torch.logsumexp(s.masked_fill(~tm, float("-inf")), dim=-1)
    np.testing.assert_allclose(L, lse.numpy(), rtol=0, atol=1e-12)


def test_kv_lens_equal_sdpa_on_sliced_keys():
    w = _problem(43, 2, 2, 2, 64, 128, 32, 32, 32, 1.0)
    ones = torch.ones(2, 2, 2, 4, dtype=torch.uint8)
    lens = [77, 128]
    O, L = OA.dense_masked(w.q, w.k, w.v, ones, 32, 32, kv_lens=lens)
    for b, n in enumerate(lens):
        ref = F.scaled_dot_product_attention(w.q[b:b + 1].double(), w.k[b:b + 1, :, :n].double(),
                                             w.v[b:b + 1, :, :n].double())
        np.testing.assert_allclose(O[b:b + 1], ref.numpy(), rtol=0, atol=1e-12)


def test_kv_len_zero_gives_empty_rows():
    w = _problem(44, 1, 1, 1, 32, 64, 32, 32, 32, 1.0)
    ones = torch.ones(1, 1, 1, 2, dtype=torch.uint8)
    O, L = OA.block_gather(w.q, w.k, w.v, ones, 32, 32, kv_lens=[0])
    assert np.all(O == 0.0) and np.all(np.isneginf(L))


@pytest.mark.parametrize("bq,bk", [(32, 32), (64, 32), (32, 64)])
def test_element_mask_forms_agree(bq, bk):
    w = _problem(45, 2, 2, 1, 128, 256, 32, bq, bk, 0.6)
    lens = [200, 131]
    O1, L1 = OA.dense_masked(w.q, w.k, w.v, w.mask, bq, bk, causal=True, kv_lens=lens)
    O2, L2 = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk, causal=True, kv_lens=lens)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(L1), np.isneginf(L2))
    fin = np.isfinite(L1)
    np.testing.assert_allclose(L1[fin], L2[fin], rtol=0, atol=1e-12)
