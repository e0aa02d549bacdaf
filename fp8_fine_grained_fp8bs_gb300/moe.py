"""Expert-parallel MoE dispatch (FP8) and combine (BF16) around the FP8
expert GEMMs.

DeepSeek-V3 "Infrastructure" §3.3.3, low-precision communication: the
activations before the MoE up-projection are quantised to FP8 (1x128 groups
with power-of-two scales) before the dispatch, so what crosses between GPUs is
E4M3 codes plus one float32 scale per 128 channels, and the expert GEMMs
consume them as they arrive; the combine after the down-projection moves and
sums BF16 values.  The page on communication/computation fusion (DeepEP)
describes the same dispatch/combine pair as all-to-all exchanges between the
ranks holding the experts.

Layout: E experts over `world` ranks, E / world per rank (expert e on rank
e // (E/world), local index e % (E/world)).  One rank's routing is topk
[T, k] (global expert ids, each token's k experts distinct) and gate weights
[T, k].

  * MoePlan (sender side): the (token, slot) pairs sorted by expert id,
    stably, so by (destination rank, local expert, token, slot); the rows sent
    to each rank; where each pair's expert output comes back.
  * RecvPlan (receiver side, from the counts every sender sends): the
    received rows arrive by source rank, each source's rows by local expert;
    the local experts' segments gather them expert by expert, each padded with
    zero rows to a multiple of 128 (the grouped GEMM's rule), and the outputs
    go back in the order the rows came.

The plans are host index arithmetic.  The data movement runs in the CUDA
library (fp8bs_scatter_q_rows, fp8bs_gather_q_rows, fp8bs_gather_bf16_rows,
fp8bs_moe_combine) and the exchanges in torch.distributed (NCCL between
GPUs); with one rank there is no exchange, and dispatch and combine each take
one launch that moves the tokens (or the expert rows) through the composed
indices.  The movement and exchange steps are parameters of dispatch() and
combine() so that the exchange protocol can be exercised with other
implementations of them.
"""
from __future__ import annotations

import numpy as np

PAD = 128


class MoePlan:
    """Sender side of the exchange for one rank's routing."""

    def __init__(self, topk, num_experts: int, world: int):
        topk = np.asarray(topk, dtype=np.int64)
        if topk.ndim != 2:
            raise ValueError("topk must be [tokens, k]")
        if num_experts % world != 0:
            raise ValueError("the experts must divide evenly over the ranks")
        if topk.size and (topk.min() < 0 or topk.max() >= num_experts):
            raise ValueError("expert id out of range")
        self.T, self.k = topk.shape
        self.E = num_experts
        self.world = world
        self.epr = num_experts // world
        flat = topk.reshape(-1)
        order = np.argsort(flat, kind="stable")           # pairs by expert id, then (token, slot)
        self.send_token = (order // self.k).astype(np.int32)   # token row of each sent row
        self.send_pos = np.empty(self.T * self.k, dtype=np.int32)
        self.send_pos[order] = np.arange(order.size, dtype=np.int32)
        self.send_pos = self.send_pos.reshape(self.T, self.k)  # where pair (t, j) sits in the send order
        self.expert_counts = np.bincount(flat, minlength=num_experts).astype(np.int64)
        self.send_counts = self.expert_counts.reshape(world, self.epr).sum(axis=1)

    def counts_for(self, dst: int) -> np.ndarray:
        """Rows this rank sends to rank dst, per local expert of dst."""
        return self.expert_counts[dst * self.epr:(dst + 1) * self.epr]


class RecvPlan:
    """Receiver side: recv_counts[src][le] rows arrive from rank src for local
    expert le (in src's send order: by local expert, then token)."""

    def __init__(self, recv_counts):
        rc = np.asarray(recv_counts, dtype=np.int64)
        self.world, self.epr = rc.shape
        self.recv_counts = rc
        self.recv_per_src = rc.sum(axis=1)
        self.rows = int(rc.sum())
        src_start = np.concatenate([[0], np.cumsum(self.recv_per_src)[:-1]])
        le_start = np.concatenate([np.zeros((self.world, 1), np.int64), np.cumsum(rc, axis=1)[:, :-1]], axis=1)
        seg = rc.sum(axis=0)                                   # rows per local expert
        padded = (seg + PAD - 1) // PAD * PAD
        self.offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
        self.padded_rows = int(self.offsets[-1])
        unpack = np.full(self.padded_rows, -1, dtype=np.int32)
        back = np.empty(self.rows, dtype=np.int32)
        for le in range(self.epr):
            pos = int(self.offsets[le])
            for src in range(self.world):
                n = int(rc[src, le])
                first = int(src_start[src] + le_start[src, le])
                unpack[pos:pos + n] = np.arange(first, first + n, dtype=np.int32)
                back[first:first + n] = np.arange(pos, pos + n, dtype=np.int32)
                pos += n
        self.unpack_idx = unpack     # padded expert row -> received row (-1: zero padding)
        self.back_idx = back         # received row -> its padded expert row
        self.pad_rows = np.nonzero(unpack < 0)[0].astype(np.int32)   # the padding rows


def exchange_counts(plan: MoePlan, all_to_all=None, make_tensor=None) -> RecvPlan:
    """Every rank sends each rank the number of rows per local expert it will
    send (a [world, E/world] exchange); returns the receiver plan."""
    send = plan.expert_counts.reshape(plan.world, plan.epr)
    if plan.world == 1:
        return RecvPlan(send)
    import torch
    mk = make_tensor or (lambda a: torch.from_numpy(np.ascontiguousarray(a)))
    inp = mk(send.reshape(-1))
    out = mk(np.zeros(plan.world * plan.epr, np.int64))
    (all_to_all or _a2a)(out, inp, [plan.epr] * plan.world, [plan.epr] * plan.world)
    return RecvPlan(np.asarray(out.cpu()).reshape(plan.world, plan.epr))


def _a2a(out, inp, out_splits, in_splits):
    import torch.distributed as dist
    dist.all_to_all_single(out, inp, [int(x) for x in out_splits], [int(x) for x in in_splits])


def _idx(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def _kernel_gather_q(q, s, s_in_kb, idx, s_out_kb):
    """Library row gather of FP8 codes and scales (fp8bs_gather_q_rows)."""
    import torch
    from . import fp8bs_gather_q_rows, SCALES_KB_MAJOR, SCALES_ROW_MAJOR
    rows_in, H = q.shape
    n = int(idx.numel())
    q_out = torch.empty((n, H), dtype=torch.uint8, device=q.device)
    s_out = torch.empty((H // 128, n) if s_out_kb else (n, H // 128), dtype=torch.float32, device=q.device)
    fp8bs_gather_q_rows(q, s, rows_in, H, SCALES_KB_MAJOR if s_in_kb else SCALES_ROW_MAJOR, idx, n, q_out, s_out,
                        SCALES_KB_MAJOR if s_out_kb else SCALES_ROW_MAJOR)
    return q_out, s_out


def _kernel_scatter_q(q, s, s_in_kb, pos, zero_rows, rows_out, s_out_kb):
    """Library row scatter of FP8 codes and scales (fp8bs_scatter_q_rows):
    row r goes to out rows pos[r, :]; zero_rows are filled with zeros."""
    import torch
    from . import fp8bs_scatter_q_rows, SCALES_KB_MAJOR, SCALES_ROW_MAJOR
    rows_in, H = q.shape
    k = int(pos.shape[1])
    q_out = torch.empty((rows_out, H), dtype=torch.uint8, device=q.device)
    s_out = torch.empty((H // 128, rows_out) if s_out_kb else (rows_out, H // 128), dtype=torch.float32,
                        device=q.device)
    n_zero = int(zero_rows.numel()) if zero_rows is not None else 0
    fp8bs_scatter_q_rows(q, s, rows_in, H, SCALES_KB_MAJOR if s_in_kb else SCALES_ROW_MAJOR, pos, k,
                         zero_rows if n_zero else None, n_zero, rows_out, q_out, s_out,
                         SCALES_KB_MAJOR if s_out_kb else SCALES_ROW_MAJOR)
    return q_out, s_out


def _kernel_gather_bf16(y, idx):
    import torch
    from . import fp8bs_gather_bf16_rows
    n = int(idx.numel())
    out = torch.empty((n, y.shape[1]), dtype=y.dtype, device=y.device)
    fp8bs_gather_bf16_rows(y, y.shape[0], y.shape[1], idx, n, out)
    return out


def _kernel_combine(y, idx, w):
    import torch
    from . import fp8bs_moe_combine
    T, k = idx.shape
    out = torch.empty((T, y.shape[1]), dtype=y.dtype, device=y.device)
    fp8bs_moe_combine(y, y.shape[0], y.shape[1], idx, w, T, k, out)
    return out


def dispatch(xq, sx, plan: MoePlan, recv: RecvPlan, gather_q=None, scatter_q=None, all_to_all=None, to_index=None):
    """FP8 dispatch: xq [T, H] E4M3 codes and sx [H/128, T] (kb-major) scales of
    this rank's tokens -> the local experts' rows (q [padded_rows, H], s
    [H/128, padded_rows] kb-major), padded segments at recv.offsets.

    Pack (each token row read once and written to its send positions, scales
    row-major so each row's scales travel with it), exchange codes and scales,
    unpack into the expert segments.  With one rank the tokens are scattered
    straight into the segments (send position -> expert row composed) and the
    padding rows zeroed in the same launch."""
    sc = scatter_q or _kernel_scatter_q
    g = gather_q or _kernel_gather_q
    ix = to_index or (lambda a: _idx(a, xq.device))
    if plan.world == 1:
        return sc(xq, sx, True, ix(recv.back_idx[plan.send_pos]), ix(recv.pad_rows), recv.padded_rows, True)
    R = int(plan.send_counts.sum())
    send_q, send_s = sc(xq, sx, True, ix(plan.send_pos), None, R, False)
    recv_q = send_q.new_empty((recv.rows, send_q.shape[1]))
    recv_s = send_s.new_empty((recv.rows, send_s.shape[1]))
    (all_to_all or _a2a)(recv_q, send_q, recv.recv_per_src, plan.send_counts)
    (all_to_all or _a2a)(recv_s, send_s, recv.recv_per_src, plan.send_counts)
    return g(recv_q, recv_s, False, ix(recv.unpack_idx), True)


def combine(y, weights, plan: MoePlan, recv: RecvPlan, gather_bf16=None, combine_rows=None, all_to_all=None,
            to_index=None, to_weights=None):
    """BF16 combine: y [padded_rows, N] the local experts' BF16 outputs ->
    out [T, N] = sum_j w[t, j] * (output of token t's j-th expert), for this
    rank's tokens.  The outputs go back in received order, through the
    reverse exchange, and are summed with the gate weights."""
    import torch
    gb = gather_bf16 or _kernel_gather_bf16
    cb = combine_rows or _kernel_combine
    ix = to_index or (lambda a: _idx(a, y.device))
    w = to_weights(weights) if to_weights else torch.as_tensor(np.ascontiguousarray(weights, np.float32),
                                                                  device=y.device)
    if plan.world == 1:
        # no exchange: each (token, slot) reads its expert row in place
        return cb(y, ix(recv.back_idx[plan.send_pos]), w)
    back = gb(y, ix(recv.back_idx))
    ret = back.new_empty((int(plan.send_counts.sum()), back.shape[1]))
    (all_to_all or _a2a)(ret, back, plan.send_counts, recv.recv_per_src)
    return cb(ret, ix(plan.send_pos), w)
