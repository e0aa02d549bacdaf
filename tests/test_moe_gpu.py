"""MoE dispatch (FP8) and combine (BF16) kernels on the GPU.

DeepSeek-V3 §3.3.3, low-precision communication: the dispatched rows are
E4M3 codes with their power-of-two 1x128 scales, the combine sums BF16
expert outputs with the gate weights.  The row gathers and the scatter must
move codes, scales and BF16 values bit for bit (numpy computes the expected
rows from the same index arrays); the combine must be within 1 BF16 ulp of
the oracle's correctly rounded weighted sum.  With one rank the exchanges are the
identity, so dispatch -> grouped GEMM -> combine runs whole here and is
checked against the oracle.
"""
import numpy as np
import pytest

import oracle
from fp8_fine_grained_fp8bs_gb300 import moe, synth
from _gpu import require_gpu, to_dev, to_dev_bf16, to_host
from _parity import check_bf16

pytestmark = pytest.mark.gpu


def _np_rows(a, idx):
    out = np.zeros((len(idx),) + a.shape[1:], a.dtype)
    ok = (idx >= 0) & (idx < a.shape[0])
    out[ok] = a[idx[ok]]
    return out


@pytest.mark.parametrize("s_in_kb", [True, False])
@pytest.mark.parametrize("s_out_kb", [True, False])
def test_gather_q_rows(s_in_kb, s_out_kb):
    torch, fp8bs = require_gpu()
    rows_in, H, rows_out = 300, 640, 517
    rng = np.random.default_rng(1)
    q = rng.integers(0, 256, (rows_in, H), dtype=np.uint8)
    s = rng.standard_normal((rows_in, H // 128)).astype(np.float32)
    idx = rng.integers(-3, rows_in + 2, rows_out).astype(np.int32)    # padding and out-of-range rows too
    s_dev = to_dev(np.ascontiguousarray(s.T) if s_in_kb else s)
    q_out = torch.empty((rows_out, H), dtype=torch.uint8, device="cuda:0")
    s_out = torch.empty((H // 128, rows_out) if s_out_kb else (rows_out, H // 128), dtype=torch.float32,
                        device="cuda:0")
    fp8bs.fp8bs_gather_q_rows(to_dev(q), s_dev, rows_in, H, 0 if s_in_kb else 1, to_dev(idx), rows_out, q_out, s_out,
                              0 if s_out_kb else 1)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(q_out), _np_rows(q, idx))
    got_s = to_host(s_out)
    got_s = got_s.T if s_out_kb else got_s
    assert np.array_equal(got_s.view(np.uint32), _np_rows(s, idx).view(np.uint32))


@pytest.mark.parametrize("s_in_kb", [True, False])
@pytest.mark.parametrize("s_out_kb", [True, False])
def test_scatter_q_rows(s_in_kb, s_out_kb):
    """Each input row to its k destinations, listed rows zeroed, the rest of
    the output untouched; destinations out of range are skipped."""
    torch, fp8bs = require_gpu()
    rows_in, H, k, rows_out = 300, 640, 3, 1000
    rng = np.random.default_rng(3)
    q = rng.integers(0, 256, (rows_in, H), dtype=np.uint8)
    s = rng.standard_normal((rows_in, H // 128)).astype(np.float32)
    perm = rng.permutation(rows_out).astype(np.int32)
    pos = perm[:rows_in * k].reshape(rows_in, k).copy()
    pos[::17, 1] = -1                   # skipped
    pos[::23, 2] = rows_out + 5         # out of range: skipped
    zero_rows = np.concatenate([perm[rows_in * k:rows_in * k + 60], [-1, rows_out]]).astype(np.int32)
    untouched = perm[rows_in * k + 60:]
    q_out = torch.full((rows_out, H), 0x5A, dtype=torch.uint8, device="cuda:0")
    s_out = torch.full((H // 128, rows_out) if s_out_kb else (rows_out, H // 128), 7.0, dtype=torch.float32,
                       device="cuda:0")
    s_dev = to_dev(np.ascontiguousarray(s.T) if s_in_kb else s)
    fp8bs.fp8bs_scatter_q_rows(to_dev(q), s_dev, rows_in, H, 0 if s_in_kb else 1, to_dev(pos), k,
                               to_dev(zero_rows), len(zero_rows), rows_out, q_out, s_out, 0 if s_out_kb else 1)
    torch.cuda.synchronize()
    exp_q = np.full((rows_out, H), 0x5A, np.uint8)
    exp_s = np.full((rows_out, H // 128), 7.0, np.float32)
    for r in range(rows_in):
        for d in pos[r]:
            if 0 <= d < rows_out:
                exp_q[d], exp_s[d] = q[r], s[r]
    for d in zero_rows:
        if 0 <= d < rows_out:
            exp_q[d], exp_s[d] = 0, 0.0
    got_s = to_host(s_out)
    got_s = got_s.T if s_out_kb else got_s
    assert np.array_equal(to_host(q_out), exp_q)
    assert np.array_equal(got_s.view(np.uint32), exp_s.view(np.uint32))
    assert np.all(to_host(q_out)[untouched] == 0x5A)


def test_scatter_q_rows_edge_cases():
    """k = 1 (a permutation), no source rows with padding rows only, and a
    single 128-column group."""
    torch, fp8bs = require_gpu()
    H = 128
    rng = np.random.default_rng(4)
    q = rng.integers(0, 256, (64, H), dtype=np.uint8)
    s = rng.standard_normal((64, 1)).astype(np.float32)
    pos = rng.permutation(64).astype(np.int32).reshape(64, 1)
    q_out = torch.empty((64, H), dtype=torch.uint8, device="cuda:0")
    s_out = torch.empty((1, 64), dtype=torch.float32, device="cuda:0")
    fp8bs.fp8bs_scatter_q_rows(to_dev(q), to_dev(s), 64, H, 1, to_dev(pos), 1, None, 0, 64, q_out, s_out, 0)
    torch.cuda.synchronize()
    exp_q = np.empty_like(q)
    exp_q[pos[:, 0]] = q
    exp_s = np.empty(64, np.float32)
    exp_s[pos[:, 0]] = s[:, 0]
    assert np.array_equal(to_host(q_out), exp_q)
    assert np.array_equal(to_host(s_out)[0].view(np.uint32), exp_s.view(np.uint32))
    # only padding rows: rows 3 and 17 zeroed, the rest untouched
    q_out.fill_(0x33)
    s_out.fill_(2.0)
    fp8bs.fp8bs_scatter_q_rows(None, None, 0, H, 0, None, 1, to_dev(np.array([3, 17], np.int32)), 2, 64, q_out,
                               s_out, 0)
    torch.cuda.synchronize()
    got_q, got_s = to_host(q_out), to_host(s_out)[0]
    assert np.all(got_q[[3, 17]] == 0) and np.all(got_s[[3, 17]] == 0.0)
    assert np.all(np.delete(got_q, [3, 17], axis=0) == 0x33) and np.all(np.delete(got_s, [3, 17]) == 2.0)
    assert fp8bs.fp8bs_get_device_status() == 0


def test_gather_bf16_rows():
    torch, fp8bs = require_gpu()
    y = synth.normal_bf16((250, 1032), 2.0, 3, 1)
    idx = np.random.default_rng(2).integers(-1, 250, 400).astype(np.int32)
    out = torch.empty((400, 1032), dtype=torch.bfloat16, device="cuda:0")
    fp8bs.fp8bs_gather_bf16_rows(to_dev_bf16(y), 250, 1032, to_dev(idx), 400, out)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, _np_rows(y, idx))


@pytest.mark.parametrize("k", [1, 2, 8, 13])
def test_combine_vs_oracle(k):
    torch, fp8bs = require_gpu()
    R, N, T = 700, 2048, 300
    y = synth.normal_bf16((R, N), 1.5, 4, 1)
    rng = np.random.default_rng(k)
    idx = rng.integers(0, R, (T, k)).astype(np.int32)
    idx[::7, 0] = -1                                      # a missing expert contributes nothing
    w = synth.moe_gate_weights(seed=k, tokens=T, top_k=k)
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda:0")
    fp8bs.fp8bs_moe_combine(to_dev_bf16(y), R, N, to_dev(idx), to_dev(w), T, k, out)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_get_device_status() == 0
    _, Y, A = oracle.moe_combine(oracle.bf16_bits_to_f32(y), idx, w)
    check_bf16(to_host(out), Y, A, f"combine k={k}")


def _single_rank_layer(torch, fp8bs, tokens, E, top_k, H, N, seed):
    """One rank: quantise (power-of-two scales), dispatch, gate/up grouped GEMM
    (BF16 out), combine; returns the device results and the host inputs."""
    x = synth.normal_bf16((tokens, H), 1.0, seed, synth.TID_X, outliers=True)
    topk = synth.moe_routing(seed=seed, tokens=tokens, experts=E, top_k=top_k)
    gw = synth.moe_gate_weights(seed=seed, tokens=tokens, top_k=top_k)
    w = synth.normal_bf16((E, N, H), 0.02, seed, synth.TID_W_GATE_UP)
    xq, sx = fp8bs.quantize_act(to_dev_bf16(x), pow2=True)
    plan = moe.MoePlan(topk, E, 1)
    recv = moe.exchange_counts(plan)
    q_exp, s_exp = moe.dispatch(xq, sx, plan, recv)
    wq = torch.empty((E, N, H), dtype=torch.uint8, device="cuda:0")
    sw = torch.empty((E, N // 128, H // 128), dtype=torch.float32, device="cuda:0")
    for e in range(E):
        fp8bs.fp8bs_quantize_weight(to_dev_bf16(w[e]), N, H, H, wq[e], sw[e])
    y = fp8bs.grouped_gemm(q_exp, s_exp, to_dev(recv.offsets.astype(np.int32)), wq, sw, out_dtype=torch.bfloat16)
    out = moe.combine(y, gw, plan, recv)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_get_device_status() == 0
    return dict(x=x, topk=topk, gw=gw, w=w, plan=plan, recv=recv, q_exp=q_exp, s_exp=s_exp, y=y, out=out)


def test_single_rank_dispatch_gemm_combine():
    torch, fp8bs = require_gpu()
    E, H, N = 6, 512, 256
    r = _single_rank_layer(torch, fp8bs, tokens=200, E=E, top_k=3, H=H, N=N, seed=5)
    plan, recv = r["plan"], r["recv"]
    # dispatch: the oracle's codes and scales of each token, in the experts' padded segments
    qa, sa = oracle.quantize_act_1x128(r["x"], pow2=True)
    src = np.where(recv.unpack_idx >= 0, plan.send_token[np.maximum(recv.unpack_idx, 0)], -1)
    assert np.array_equal(to_host(r["q_exp"]), _np_rows(qa, src))
    assert np.array_equal(to_host(r["s_exp"]).T.view(np.uint32), _np_rows(sa, src).view(np.uint32))
    # the experts' GEMM on what arrived
    qb = np.stack([oracle.quantize_weight_128x128(r["w"][e])[0] for e in range(E)])
    sb = np.stack([oracle.quantize_weight_128x128(r["w"][e])[1] for e in range(E)])
    Y, T = oracle.grouped_gemm_block_scaled(_np_rows(qa, src), _np_rows(sa, src), recv.offsets, qb, sb)
    y = to_host(r["y"])
    check_bf16(y, Y, T, "expert GEMM on dispatched rows")
    # combine of the GEMM's BF16 outputs (exact inputs to the combine)
    _, Yc, Ac = oracle.moe_combine(y[recv.back_idx], plan.send_pos, r["gw"])
    check_bf16(to_host(r["out"]), Yc, Ac, "combine")


def test_full_size_dispatch_and_combine_sampled():
    """8192 tokens, top-8 of 32 experts, hidden 7168 (the MoE workload's
    routing): dispatch moves every code and scale to its place; the combine of
    the gate/up GEMM's output, checked on sampled tokens."""
    torch, fp8bs = require_gpu()
    E, H, N = 32, 7168, 256
    r = _single_rank_layer(torch, fp8bs, tokens=8192, E=E, top_k=8, H=H, N=N, seed=0)
    plan, recv = r["plan"], r["recv"]
    qa, sa = oracle.quantize_act_1x128(r["x"], pow2=True)
    src = np.where(recv.unpack_idx >= 0, plan.send_token[np.maximum(recv.unpack_idx, 0)], -1)
    assert np.array_equal(to_host(r["q_exp"]), _np_rows(qa, src))
    assert np.array_equal(to_host(r["s_exp"]).T.view(np.uint32), _np_rows(sa, src).view(np.uint32))
    y = to_host(r["y"])
    toks = np.unique(np.concatenate([np.arange(0, 8192, 97), [8191]]))
    _, Yc, Ac = oracle.moe_combine(y[recv.back_idx], plan.send_pos[toks], r["gw"][toks])
    check_bf16(to_host(r["out"])[toks], Yc, Ac, "combine, full-size routing")
