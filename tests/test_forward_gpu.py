"""GPU forward (tcgen05/TMA kernel, through the C ABI) vs the fp64 oracle on the
same seeded bf16 inputs."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from block_sparse_attention_plan_gb300 import workloads as W
from compare import assert_attention_close

pytestmark = pytest.mark.gpu


def run_gpu(bsa, w, scale=None):
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda(), scale=scale)
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    return o, lse


@pytest.mark.parametrize("name", list(W.SMALL_CONFIGS))
def test_forward_small_configs(bsa, name):
    w = W.make_workload(name)
    o, lse = run_gpu(bsa, w)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, w.bq, w.bk)
    assert_attention_close(o, lse, O, L, name, record=True)


@pytest.mark.parametrize("bq,bk,d,g", [
    (128, 128, 128, 1), (128, 128, 64, 2), (64, 64, 128, 1), (64, 64, 64, 4), (32, 32, 64, 1),
    (32, 128, 128, 2), (128, 32, 64, 1), (64, 32, 128, 1), (256, 128, 64, 1), (128, 256, 128, 2),
    (256, 256, 64, 1), (32, 256, 128, 1),
])
def test_forward_mappings(bsa, bq, bk, d, g):
    w = W.random_problem(31 + bq + bk + d, 1, 4, 4 // g, 1024, 1536, d, bq, bk, 0.3)
    w.mask[0, 1, 0, :] = 0   # an empty logical q-block row
    o, lse = run_gpu(bsa, w)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk)
    assert_attention_close(o, lse, O, L, f"bq={bq} bk={bk} d={d} g={g}")


@pytest.mark.parametrize("d", [64, 128])
def test_forward_all_ones_and_all_zero(bsa, d):
    w = W.random_problem(5, 1, 2, 2, 512, 768, d, 128, 128, 1.1)
    o, lse = run_gpu(bsa, w)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128)
    assert_attention_close(o, lse, O, L, "all ones")
    w.mask.zero_()
    o, lse = run_gpu(bsa, w)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_forward_scale_override_and_long_rows(bsa):
    w = W.random_problem(9, 1, 2, 2, 256, 8192, 128, 128, 128, 0.9)
    o, lse = run_gpu(bsa, w, scale=0.05)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128, scale=0.05)
    assert_attention_close(o, lse, O, L, "scale")


def test_forward_large_logits_rescale(bsa):
    # Scores growing along the key axis (by about 60 in log2 units over the
    # sequence) force the running max past the lazy-rescale threshold (16 log2
    # units) several times.
    w = W.random_problem(12, 1, 2, 2, 256, 4096, 128, 128, 128, 1.1)
    ramp = torch.linspace(0.2, 3.0, 4096).view(1, 1, 4096, 1)
    w.k = (w.k.float() * ramp).to(torch.bfloat16)
    w.q = (w.q.float() * 4.0).to(torch.bfloat16)
    o, lse = run_gpu(bsa, w)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128)
    assert_attention_close(o, lse, O, L, "rescale")


# Control word holding the number of plan rows the bounded pass queued for
# the exact pass (index 3 of the plan's control words).
FALLBACK_COUNT = 3


def test_forward_loose_bound_rows_take_exact_pass(bsa):
    # Heads 0-1 (K/V head 0): a large query component on channel 0 and a large
    # key component on channel 1 make |q||k| (the row bound) exceed every
    # score by thousands of log2 units, so the bounded pass underflows there
    # and must hand those rows to the exact pass; heads 2-3 stay ordinary.
    w = W.random_problem(21, 1, 4, 2, 512, 1024, 128, 128, 128, 0.7)
    q, k = w.q.float(), w.k.float()
    q[:, :2, :, 0] = 150.0
    k[:, :1, :, 1] = 150.0
    w.q, w.k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda())
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    queued = int(p.control()[FALLBACK_COUNT].item())
    rows_h01 = 2 * (512 // 128)
    nonempty_h01 = int((w.mask[0, :2].reshape(2, 4, -1).sum(-1) > 0).sum())
    assert nonempty_h01 <= queued <= rows_h01, (queued, nonempty_h01)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 128, 128)
    assert_attention_close(o, lse, O, L, "loose bound")


@pytest.mark.parametrize("name", ["video_dit_small", "chunked_prefill_small", "regular_small",
                                  "long_video_dit_small"])
def test_forward_bounded_pass_queues_nothing_on_workloads(bsa, name):
    # On the benchmark-shaped inputs the row bound stays close enough to the
    # scores that no row should need the exact pass.
    w = W.make_workload(name)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda())
    assert bsa.sync_status(p)[0] == 0
    assert int(p.control()[FALLBACK_COUNT].item()) == 0


@pytest.mark.parametrize("d", [64, 128])
def test_forward_output_16_byte_aligned(bsa, d):
    """An O whose base is 16- but not 32-byte aligned (the alignment the C ABI
    asks for) is written with 16-byte stores instead of 32-byte ones: the same
    values, bit for bit."""
    w = W.random_problem(13 + d, 1, 2, 2, 512, 768, d, 128, 128, 0.5)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, 1)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o1, l1 = bsa.forward(p, q, k, v)
    buf = torch.empty(o1.numel() + 8, dtype=torch.bfloat16, device="cuda")
    o2 = buf[8:].view(o1.shape)
    assert o1.data_ptr() % 32 == 0 and o2.data_ptr() % 32 == 16
    _, l2 = bsa.forward(p, q, k, v, out=o2)
    assert bsa.sync_status(p)[0] == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_forward_repeat_and_plan_reuse(bsa):
    w = W.make_workload("video_dit_small")
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, 1)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o1, l1 = bsa.forward(p, q, k, v)
    o2, l2 = bsa.forward(p, q, k, v)
    assert bsa.sync_status(p)[0] == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["video_dit", "chunked_prefill", "regular"])
def test_forward_full_configs(bsa, name):
    w = W.make_workload(name)
    o, lse = run_gpu(bsa, w)
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, w.bq, w.bk)
    assert_attention_close(o, lse, O, L, name, record=True)


@pytest.mark.slow
def test_forward_long_video_sampled(bsa):
    w = W.make_workload("long_video_dit")
    o, lse = run_gpu(bsa, w)
    H, NQB = w.Hq, w.mask.shape[2]
    samples = [(0, h, qb) for h in range(H) for qb in range(h % 16, NQB, 16)] + [(0, 0, NQB - 1), (0, 39, NQB - 1)]
    ref = OA.sampled_qblocks(w.q, w.k, w.v, w.mask, w.bq, w.bk, samples)
    og = torch.cat([o[0, h, qb * 128:(qb + 1) * 128] for (_, h, qb) in samples]).cpu()
    lg = torch.cat([lse[0, h, qb * 128:(qb + 1) * 128] for (_, h, qb) in samples]).cpu()
    Oref = np.concatenate([ref[s][0] for s in samples])
    Lref = np.concatenate([ref[s][1] for s in samples])
    assert_attention_close(og, lg, Oref, Lref, "long_video_dit (sampled q-blocks)", record=True)
    assert torch.all(o[0, :, -128:] == 0) and torch.all(torch.isneginf(lse[0, :, -128:]))



@pytest.mark.parametrize("bq,bk,d", [(32, 32, 64), (64, 128, 128), (32, 256, 128)])
def test_forward_remapped_plan_vs_oracle(bsa, bq, bk, d):
    # Planes regrouped by the plan (q-units of a tile strided through the
    # head): Q loads per q-unit, O/LSE rows written back to their positions.
    w = W.random_problem(61 + bq, 2, 4, 4, 1024, 1024, d, bq, bk, 0.05)
    NQB, NKB = 1024 // bq, 1024 // bk
    x = torch.arange(NQB).view(NQB, 1)
    kb = torch.arange(NKB).view(1, NKB)
    w.mask[:, 1] |= ((kb % 4) == (x % 4)).to(torch.uint8)
    w.mask[:, 2] |= ((kb % 2) == (x % 2)).to(torch.uint8)
    p = bsa.plan(w.mask.cuda(), bq, bk, 1, flags=bsa.PLAN_REMAP)
    assert max(p.arrays()["plane_sigma"].tolist()) > 1
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda())
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk)
    assert_attention_close(o, lse, O, L, f"remapped {bq}x{bk} d{d}")


def test_forward_remapped_plan_causal_kv_lens(bsa):
    w = W.random_problem(71, 2, 2, 2, 512, 1024, 64, 64, 64, 0.3)
    NQB, NKB = 512 // 64, 1024 // 64
    x = torch.arange(NQB).view(NQB, 1)
    kb = torch.arange(NKB).view(1, NKB)
    w.mask[:, 0] |= ((kb % 2) == (x % 2)).to(torch.uint8)
    lens = torch.tensor([1000, 700], dtype=torch.int32)
    p = bsa.plan(w.mask.cuda(), 64, 64, 1, flags=bsa.PLAN_REMAP)
    o, lse = bsa.forward(p, w.q.cuda(), w.k.cuda(), w.v.cuda(), causal=True, kv_lens=lens.cuda())
    st, det = bsa.sync_status(p)
    assert st == 0, (st, hex(det))
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, 64, 64, causal=True, kv_lens=lens.tolist())
    assert_attention_close(o, lse, O, L, "remapped causal kv_lens")


@pytest.mark.parametrize("name", ["video_dit_small", "chunked_prefill_small"])
def test_forward_in_stages_equals_forward(bsa, name):
    w = W.make_workload(name)
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o1, l1 = bsa.forward(p, q, k, v)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    for st in (bsa.STAGE_PREPARE, bsa.STAGE_BOUNDED, bsa.STAGE_EXACT):
        bsa.forward(p, q, k, v, out=o2, lse=l2, stages=st)
    assert bsa.sync_status(p)[0] == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = torch.empty_like(o1), torch.empty_like(l1)
    bsa.forward(p, q, k, v, out=o3, lse=l3, stages=bsa.STAGE_PREPARE | bsa.STAGE_BOUNDED)
    bsa.forward(p, q, k, v, out=o3, lse=l3, stages=bsa.STAGE_EXACT)
    assert torch.equal(o1, o3)
    for bad in (0, 0x20):
        with pytest.raises(bsa.BsaError):
            bsa.forward(p, q, k, v, stages=bad)


def test_key_norm_stage_beside_plan_creation(bsa):
    # The key-norm stage reads only K: enqueued on a side stream that starts
    # with the plan kernels (not after them), then the rest of the forward.
    w = W.make_workload("chunked_prefill_small")
    q, k, v, mask = w.q.cuda(), w.k.cuda(), w.v.cuda(), w.mask.cuda()
    p0 = bsa.plan(mask, w.bq, w.bk, w.gqa_group)
    o_ref, l_ref = bsa.forward(p0, q, k, v)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    fork = torch.cuda.Event()
    for _ in range(3):
        fork.record(main)
        p = bsa.plan(mask, w.bq, w.bk, w.gqa_group)
        side.wait_event(fork)
        o, lse = torch.empty_like(o_ref), torch.empty_like(l_ref)
        bsa.forward(p, q, k, v, out=o, lse=lse, stages=bsa.STAGE_KNORM, stream=side)
        main.wait_stream(side)
        bsa.forward(p, q, k, v, out=o, lse=lse,
                    stages=bsa.STAGE_ROWBOUND | bsa.STAGE_BOUNDED | bsa.STAGE_EXACT)
        assert bsa.sync_status(p)[0] == 0
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


# Split weights (hi + lo bf16 terms): forced on every row, or chosen by the
# kernel for rows whose K/V units hold a |v| above 8.
@pytest.mark.parametrize("bq,bk,d,g", [(128, 128, 128, 1), (64, 64, 128, 2), (32, 32, 64, 1),
                                       (256, 128, 64, 1), (128, 32, 128, 1)])
def test_forward_split_weights_vs_oracle(bsa, bq, bk, d, g):
    w = W.random_problem(81 + bq + d, 1, 4, 4 // g, 1024, 1536, d, bq, bk, 0.3)
    w.mask[0, 2, 1, :] = 0
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    p = bsa.plan(w.mask.cuda(), bq, bk, g)
    o, lse = bsa.forward(p, q, k, v, split=True)
    assert bsa.sync_status(p)[0] == 0
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk)
    assert_attention_close(o, lse, O, L, f"split {bq}x{bk} d{d} g{g}")
    # V with a few large channels: the default path splits by itself
    vbig = w.v.float()
    vbig[:, :, :, :3] *= 16.0
    w.v = vbig.to(torch.bfloat16)
    o2, l2 = bsa.forward(p, q, k, w.v.cuda())
    o3, l3 = bsa.forward(p, q, k, w.v.cuda(), split=True)
    assert bsa.sync_status(p)[0] == 0
    O, L = OA.block_gather(w.q, w.k, w.v, w.mask, bq, bk)
    assert_attention_close(o2, l2, O, L, f"large V {bq}x{bk} d{d} g{g}")
    assert torch.equal(o2, o3) and torch.equal(l2, l3)


def test_forward_split_rows_are_the_large_value_heads(bsa):
    # Outlier channels (x8) put |v| far above 8 in every unit of the heads
    # that have one: those rows are computed with split weights by default
    # (bit-identical to forcing it), the other heads' rows are not.
    w = W.make_workload("long_video_dit_small")
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    p = bsa.plan(w.mask.cuda(), w.bq, w.bk, w.gqa_group)
    o1, l1 = bsa.forward(p, q, k, v)
    o2, l2 = bsa.forward(p, q, k, v, split=True)
    assert bsa.sync_status(p)[0] == 0
    big = (w.v.float().abs().amax(dim=(2, 3)) > 8.0)[0].tolist()
    assert any(big) and not all(big)
    for h in range(w.Hq):
        same = torch.equal(o1[0, h], o2[0, h]) and torch.equal(l1[0, h], l2[0, h])
        if big[h // w.gqa_group]:
            assert same, h
