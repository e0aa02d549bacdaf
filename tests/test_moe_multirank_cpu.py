"""Expert-parallel MoE layer over two gloo ranks on the CPU: FP8 dispatch,
expert GEMMs, BF16 combine (DeepSeek-V3 §3.3.3, low-precision
communication: the activations are quantised to FP8 with power-of-two
scales before the dispatch, the experts' FP8 GEMMs consume what arrives, and
the combine moves and sums BF16).

Each rank routes its own tokens (top-2 of 4 experts, 2 experts per rank),
plans the exchange (fp8_fine_grained_fp8bs_gb300.moe), exchanges the counts,
the E4M3 codes with their scales, and the BF16 expert outputs with gloo
all-to-alls, and computes the expert GEMMs, SwiGLU and combine with the
oracle; the row copies around the exchanges are numpy here (the library's
scatter and gather kernels are checked on the GPU).  Every row's arithmetic depends on
that row only, so the two ranks' outputs must equal the single-process
layer over all tokens bit for bit.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

H, I, E, TOPK, T = 256, 128, 4, 2, 96


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _np_gather_q(q, s, s_in_kb, idx, s_out_kb):
    qn, sn = q.numpy(), s.numpy()
    rows = sn.T if s_in_kb else sn
    ok = (idx >= 0) & (idx < qn.shape[0])
    qo = np.zeros((len(idx), qn.shape[1]), np.uint8)
    so = np.zeros((len(idx), rows.shape[1]), np.float32)
    qo[ok] = qn[idx[ok]]
    so[ok] = rows[idx[ok]]
    return torch.from_numpy(qo), torch.from_numpy(np.ascontiguousarray(so.T) if s_out_kb else so)


def _np_scatter_q(q, s, s_in_kb, pos, zero_rows, rows_out, s_out_kb):
    qn, sn = q.numpy(), s.numpy()
    rows = sn.T if s_in_kb else sn
    qo = np.zeros((rows_out, qn.shape[1]), np.uint8)
    so = np.zeros((rows_out, rows.shape[1]), np.float32)
    written = np.zeros(rows_out, np.int64)
    for r in range(qn.shape[0]):
        for d in pos[r]:
            if 0 <= d < rows_out:
                qo[d] = qn[r]
                so[d] = rows[r]
                written[d] += 1
    if zero_rows is not None:
        written[np.asarray(zero_rows)] += 1
    # the planner names every out row exactly once (a token row or padding)
    assert np.all(written == 1), np.bincount(written)
    return torch.from_numpy(qo), torch.from_numpy(np.ascontiguousarray(so.T) if s_out_kb else so)


def _np_gather_bf16(y, idx):
    yn = y.numpy()
    out = np.zeros((len(idx), yn.shape[1]), yn.dtype)
    ok = idx >= 0
    out[ok] = yn[idx[ok]]
    return torch.from_numpy(out)


def _np_combine(y, idx, w):
    import oracle
    return torch.from_numpy(oracle.moe_combine(y.numpy(), idx, w)[0].astype(np.float32))


def _weights():
    import oracle
    from fp8_fine_grained_fp8bs_gb300 import synth
    wgu = synth.normal_bf16((E, 2 * I, H), 0.02, 7, synth.TID_W_GATE_UP)
    wdn = synth.normal_bf16((E, H, I), 0.02, 7, synth.TID_W_DOWN)
    gu = [oracle.quantize_weight_128x128(wgu[e]) for e in range(E)]
    dn = [oracle.quantize_weight_128x128(wdn[e]) for e in range(E)]
    return (np.stack([g[0] for g in gu]), np.stack([g[1] for g in gu]),
            np.stack([d[0] for d in dn]), np.stack([d[1] for d in dn]))


def _experts(q_exp, s_exp_kb, offsets, ids, w):
    """The experts' layer on their padded segments: gate/up GEMM (BF16 out),
    SwiGLU + 1x128 quantisation, down GEMM (BF16 out)."""
    import oracle
    from fp8_fine_grained_fp8bs_gb300 import synth
    gq, gs, dq, ds = w
    y1, _ = oracle.grouped_gemm_block_scaled(q_exp, np.ascontiguousarray(s_exp_kb.T), offsets, gq[ids], gs[ids])
    h = synth.f32_to_bf16_bits(oracle.bf16_round(y1).astype(np.float32))
    q2, s2 = oracle.swiglu_quantize_1x128(h, I)
    y2, _ = oracle.grouped_gemm_block_scaled(q2, s2, offsets, dq[ids], ds[ids])
    return oracle.bf16_round(y2).astype(np.float32)           # BF16 values, exact in float32


def _inputs(rank):
    from fp8_fine_grained_fp8bs_gb300 import synth
    x = synth.normal_bf16((T, H), 1.0, rank, synth.TID_X, outliers=True)
    topk = synth.moe_routing(seed=100 + rank, tokens=T, experts=E, top_k=TOPK)
    gw = synth.moe_gate_weights(seed=100 + rank, tokens=T, top_k=TOPK)
    return x, topk, gw


def _layer(x, topk, gw, world, rank, w):
    import oracle
    from fp8_fine_grained_fp8bs_gb300 import moe
    q, s = oracle.quantize_act_1x128(x, pow2=True)
    plan = moe.MoePlan(topk, E, world)
    recv = moe.exchange_counts(plan)
    q_exp, s_exp = moe.dispatch(torch.from_numpy(q), torch.from_numpy(np.ascontiguousarray(s.T)), plan, recv,
                                gather_q=_np_gather_q, scatter_q=_np_scatter_q, to_index=lambda a: a)
    ids = rank * plan.epr + np.arange(plan.epr)
    y = _experts(q_exp.numpy(), s_exp.numpy(), recv.offsets, ids, w)
    out = moe.combine(torch.from_numpy(y), gw, plan, recv, gather_bf16=_np_gather_bf16, combine_rows=_np_combine,
                      to_index=lambda a: a, to_weights=lambda a: a)
    return out.numpy(), recv.offsets


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out, offsets = _layer(*_inputs(rank), world, rank, _weights())
        parts = [None] * world
        dist.all_gather_object(parts, (out, offsets))
        if rank == 0:
            q.put(parts)
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_layer_equals_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    parts = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # the same layer in one process over both ranks' tokens, all experts local
    ins = [_inputs(r) for r in range(2)]
    x = np.concatenate([i[0] for i in ins])
    topk = np.concatenate([i[1] for i in ins])
    gw = np.concatenate([i[2] for i in ins])
    ref, _ = _layer(x, topk, gw, 1, 0, _weights())
    got = np.concatenate([p[0] for p in parts])
    assert got.shape == (2 * T, H)
    assert np.array_equal(got, ref)
    assert np.count_nonzero(ref) > 0.9 * ref.size
    # each rank's experts got rows from both ranks, padded to 128 per expert
    for _, offsets in parts:
        assert np.all(np.diff(offsets) % 128 == 0) and offsets[-1] > 0
