"""The MoE combine oracle and the dispatch/combine planner, on the CPU.

The combine (DeepSeek-V3 §3.3.3: kept in BF16) is out[t] = BF16(sum_j
w[t][j] * y_j[t]); pinned by hand-worked values, the one-expert identity, an
exact BF16 tie, and a planted mistake.  The planner (MoePlan / RecvPlan) is
host index arithmetic; pinned by its invariants: the send order is the pairs
sorted by expert, the counts add up, the expert segments are padded to 128,
and the way back is the inverse of the way in.
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import moe, synth


def test_combine_hand_worked():
    y = np.array([[1.0, 2.0, -0.5], [3.0, -4.0, 0.25]])
    idx = np.array([[0, 1], [1, -1]])
    w = np.array([[0.5, 0.25], [1.0, 0.5]], np.float32)
    out, exact, mag = oracle.moe_combine(y, idx, w)
    # token 0: 0.5*[1,2,-0.5] + 0.25*[3,-4,0.25] = [1.25, 0, -0.1875]; token 1: [3, -4, 0.25]
    assert np.array_equal(out, [[1.25, 0.0, -0.1875], [3.0, -4.0, 0.25]])
    assert np.array_equal(mag[0], [0.5 + 0.75, 1.0 + 1.0, 0.25 + 0.0625])


def test_combine_single_expert_is_identity_on_bf16_values():
    rng = np.random.default_rng(0)
    y = oracle.bf16_bits_to_f32(synth.normal_bf16((50, 64), 3.0, 1, 1)).astype(np.float64)
    idx = rng.permutation(50)[:, None]
    out, _, _ = oracle.moe_combine(y, idx, np.ones((50, 1), np.float32))
    assert np.array_equal(out, y[idx[:, 0]])


def test_combine_rounds_once_to_nearest_even():
    # 1 + 2^-8 is halfway between the BF16 neighbours 1 and 1 + 2^-7: ties to even -> 1;
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to even -> 1 + 2^-6
    y = np.array([[1.0], [2.0 ** -8], [3 * 2.0 ** -8]])
    w = np.ones((2, 2), np.float32)
    out, exact, _ = oracle.moe_combine(y, np.array([[0, 1], [0, 2]]), w)
    assert exact[0, 0] == 1 + 2.0 ** -8 and out[0, 0] == 1.0
    assert exact[1, 0] == 1 + 3 * 2.0 ** -8 and out[1, 0] == 1 + 2.0 ** -6


def test_combine_planted_mistake_detected():
    y = np.array([[1.0], [10.0]])
    idx = np.array([[0, 1]])
    w = np.array([[0.75, 0.25]], np.float32)
    out, _, _ = oracle.moe_combine(y, idx, w)
    swapped, _, _ = oracle.moe_combine(y, idx, w[:, ::-1])
    assert out[0, 0] == 3.25 and swapped[0, 0] != out[0, 0]


@pytest.mark.parametrize("world", [1, 2, 4])
def test_plan_invariants(world):
    E, T, k = 8, 300, 3
    topk = synth.moe_routing(seed=world, tokens=T, experts=E, top_k=k)
    plan = moe.MoePlan(topk, E, world)
    # the send order is the pairs sorted by expert id (stable: token, slot)
    sent_expert = topk.reshape(-1)[np.argsort(topk.reshape(-1), kind="stable")]
    assert np.all(np.diff(sent_expert) >= 0)
    assert np.array_equal(plan.send_token, np.argsort(topk.reshape(-1), kind="stable") // k)
    # every pair has a send position, and it points at a row of its token
    assert sorted(plan.send_pos.reshape(-1).tolist()) == list(range(T * k))
    assert np.all(plan.send_token[plan.send_pos] == np.arange(T)[:, None])
    assert plan.send_counts.sum() == T * k
    assert np.array_equal(plan.send_counts, [np.isin(topk, range(d * E // world, (d + 1) * E // world)).sum()
                                             for d in range(world)])


def test_recv_plan_padding_and_inverse():
    rc = np.array([[3, 0, 130], [1, 200, 0]])     # 2 sources x 3 local experts
    rp = moe.RecvPlan(rc)
    assert rp.rows == 334 and np.array_equal(rp.recv_per_src, [133, 201])
    assert np.array_equal(rp.offsets, [0, 128, 384, 640])          # 4 -> 128, 200 -> 256, 130 -> 256
    real = rp.unpack_idx >= 0
    assert real.sum() == rp.rows
    assert np.array_equal(rp.unpack_idx[rp.back_idx], np.arange(rp.rows))   # way back inverts way in
    # expert 0 takes source 0's first 3 rows, then source 1's first row (received row 133)
    assert rp.unpack_idx[:4].tolist() == [0, 1, 2, 133] and np.all(rp.unpack_idx[4:128] == -1)
    # expert 1 takes only source 1's rows 134..333
    assert rp.unpack_idx[128:328].tolist() == list(range(134, 334))
    # expert 2 takes source 0's rows 3..132
    assert rp.unpack_idx[384:514].tolist() == list(range(3, 133))
