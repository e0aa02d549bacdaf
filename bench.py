"""Benchmark of the fine-grained FP8 hot path on GB300.

One step = the FP8 Linear forward of the dense workload with online
quantisation (DeepSeek-V3 §3.3): quantise X[4096,7168] (BF16, 1x128 tiles)
and W[7168,7168] (BF16, 128x128 blocks) in one launch, block-scaled FP8
GEMM Y = X W^T with BF16 output.  ``value`` is the step's GEMM FLOPs
(2*M*N*K) per second over the whole step, in TFLOP/s.  Measured in the same
run and reported beside it:
  * ``gemm``:     the GEMM kernel alone (CUDA events around each launch);
  * ``quantize``: the standalone 1x128 quantisation of X[16384,7168]
                  (algorithmic bytes 2 + 1 + 4/128 per element), GB/s;
  * ``roofline``: the GEMM against the FP8 dense tensor peak;
  * ``e2e``:      the step through the public API with host buffers (pinned
                  host -> device copies of X and W, device -> host copy of Y,
                  every step; steps pipelined over copy-in, compute and
                  copy-out streams with double device buffers);
  * ``cpu_baseline``: the CPU oracle on a bounded sample of the same step;
  * ``workloads``: the other configurations, each kernel timed alone: the
                  MoE grouped GEMMs (gate/up and down), dgrad, wgrad, the
                  dual-layout (1x128 + 128x1) activation quantize, the
                  weight quantize with its transposed copy, the power-of-two
                  scale quantize, the FP8 1x128 -> 128x1 re-tiling and the
                  fused SwiGLU -> 1x128 quantize of the MoE gate/up output.

Multi-GPU: every rank runs its own replica on its own batch (data
parallel, no collective on the data path); ``value`` sums all ranks' FLOPs
over the slowest rank's time ("scaling": "weak").

``--impl reference`` times the CPU oracle (the reference arm of this
method: the pages publish no code) on the same metric and prints its line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M, N, K = 4096, 7168, 7168
QM, QK = 16384, 7168
GEMM_FLOP = 2.0 * M * N * K
QUANT_BYTES = QM * QK * (2 + 1 + 4 / 128)
METRIC = "block-scaled FP8 GEMM TFLOP/s (% of FP8 peak); 1x128 quantize HBM GB/s"
WORKLOAD = ("dense fprop: quantize X[4096,7168] 1x128 + W[7168,7168] 128x128 to E4M3, "
            "block-scaled FP8 GEMM Y=X W^T BF16 out; plus standalone quantize of X[16384,7168]")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0      # nominal dense ratio (4.5 / 2.25 PFLOP/s)
NOMINAL_HBM_GBS = 7900.0 # HBM3e of one GB300, nominal
FP8_FLOP_PER_CLK_SM = 16384  # dense FP8 tcgen05 rate per SM (M=128 x N=256 x K=32 MMA in 128 cycles)


def hw_fp8_peak_tflops(sms: int, sm_mhz: float) -> float:
    """Instruction-rate FP8 peak: every SM issuing dense FP8 MMAs at its full
    rate at the given clock."""
    return sms * FP8_FLOP_PER_CLK_SM * sm_mhz * 1e6 / 1e12


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


CSRC = "fp8_fine_grained_fp8bs_gb300/csrc/"


def _traffic(kernel_key: str, *source_files: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, if
    the kernel's sources (its .cu and the device headers it includes) still
    match the ones the counters were taken on."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e:
        return None
    sha = hashlib.sha256()
    for name in source_files:
        with open(os.path.join(ROOT, name), "rb") as f:
            sha.update(f.read())
    h = sha.hexdigest()[:16]
    return e["dram_bytes_per_launch"] if e.get("source_sha256_16") == h else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.2)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _gpu_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


# ----------------------------------------------------------------- CPU oracle

def _oracle_step(x_bits, w_bits, sm_rows, sn_rows):
    import oracle
    qa, sa = oracle.quantize_act_1x128(x_bits[:sm_rows])
    qb, sb = oracle.quantize_weight_128x128(w_bits[:sn_rows])
    oracle.gemm_block_scaled(qa, sa, qb, sb)
    return 2.0 * sm_rows * sn_rows * K


def _cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def _oracle_quantize_rows(rows_bits) -> int:
    """The oracle's 1x128 quantisation of a block of rows; returns the element count."""
    import oracle
    oracle.quantize_act_1x128(rows_bits)
    return int(rows_bits.size)


def cpu_quantize_baseline(xl_bits, budget_s: float = 4.0):
    """The oracle's 1x128 quantisation of X[16384,7168], untuned, on bounded
    samples: on one core (the numpy oracle is single-threaded elementwise
    code) and on all cores (one 256-row shard per core, a process pool
    started with spawn, so no process is forked after the GPU is in use)."""
    import multiprocessing
    rows = 256
    bpe = 2 + 1 + 4 / 128
    nrows = xl_bits.shape[0]
    el, n, t0 = 0, 0, time.perf_counter()
    while True:
        r0 = (n * rows) % (nrows - rows)
        el += _oracle_quantize_rows(xl_bits[r0:r0 + rows])
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    one = el * bpe / (time.perf_counter() - t0) / 1e9
    cores = os.cpu_count() or 1
    shards = [np.ascontiguousarray(xl_bits[(i * rows) % nrows:(i * rows) % nrows + rows]) for i in range(cores)]
    with multiprocessing.get_context("spawn").Pool(cores) as pool:
        pool.map(_oracle_quantize_rows, shards)            # start-up and imports, untimed
        el_all, reps, t0 = 0, 0, time.perf_counter()
        while True:
            el_all += sum(pool.map(_oracle_quantize_rows, shards))
            reps += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt_all = time.perf_counter() - t0
    return {"unit": "GB/s", "one_core": one, "all_cores": el_all * bpe / dt_all / 1e9, "cores": cores,
            "kind": "oracle",
            "sample": f"one core: {n} blocks of 256 rows of X[16384,7168]; all cores: {reps} rounds of "
                      f"{cores} such blocks, one per process; algorithmic bytes 2 + 1 + 4/128 per element"}


def cpu_baseline(x_bits, w_bits, xl_bits=None, budget_s=12.0):
    """The oracle, untuned, on a bounded sample: X rows x W rows of the step;
    with xl_bits also the standalone 1x128 quantisation (one core and all
    cores)."""
    sm_rows, sn_rows = 512, 1024
    flop, t0, n = 0.0, time.perf_counter(), 0
    while True:
        flop += _oracle_step(x_bits, w_bits, sm_rows, sn_rows)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    out = {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": _cpu_cores(), "kind": "oracle",
           "sample": f"{n} x (quantize X[{sm_rows},7168] 1x128 + W[{sn_rows},7168] 128x128, "
                     f"GEMM {sm_rows}x{sn_rows}x7168), float64 numpy, {dt:.1f} s"}
    if xl_bits is not None:
        out["quantize_1x128"] = cpu_quantize_baseline(xl_bits)
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from fp8_fine_grained_fp8bs_gb300 import synth
    x_bits, w_bits = synth.dense_fprop(0)
    ladder = [(8, 128), (32, 128), (64, 256), (128, 256), (256, 512), (512, 1024)]
    budget = 150.0 / max(1, args.steps + args.warmup)
    pick = ladder[0]
    for cand in ladder:
        t0 = time.perf_counter()
        _oracle_step(x_bits, w_bits, *cand)
        if time.perf_counter() - t0 > budget:
            break
        pick = cand
    for _ in range(args.warmup):
        _oracle_step(x_bits, w_bits, *pick)
    t0 = time.perf_counter()
    flop = 0.0
    for _ in range(args.steps):
        flop += _oracle_step(x_bits, w_bits, *pick)
    dt = time.perf_counter() - t0
    v = flop / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample_rows": list(pick)},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": _cpu_cores(), "kind": "oracle",
                             "sample": f"each step: quantize X[{pick[0]},7168] + W[{pick[1]},7168], "
                                       f"GEMM {pick[0]}x{pick[1]}x7168"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- GPU arm

def _time_ms(fn, stream, warmup: int, reps: int) -> float:
    """Mean device time of fn() on `stream` (CUDA events around each call)."""
    import torch
    for _ in range(warmup):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


WORKLOAD_SECTIONS = ("dgrad", "wgrad", "context", "weight", "moe", "pow2")


def measure_workloads(fp8bs, synth, dev, stream, rank: int, fp8_peak: float, hbm_peak: float, warmup: int,
                      sections=WORKLOAD_SECTIONS, moe_tokens: int = 8192, moe_experts: int = 32,
                      hw_peak: float | None = None):
    """The other configurations of the path, each kernel timed alone.

    * MoE grouped fprop: 8192 tokens, top-8 of 32 experts (Zipf s=1.1),
      per-expert rows padded to 128; gate/up [67712 x 4096 x 7168] and down
      [67712 x 7168 x 2048], BF16 out.  Routing and token activations follow
      the numpy recipe; the expert weights N(0,0.02) and the down-projection
      input N(0,1) are drawn on the device by torch's seeded generator (same
      distributions, BF16-rounded) so the 1.4 G weights take no host time.
      TFLOP/s counts real (unpadded) rows.
    * dgrad dX[4096,2048] = dY[4096,7168] W[7168,2048] (FP32 out, B = the
      transposed weight copy); wgrad dW[2048,7168] = dY^T X over T = 16384
      (both 128x1 along T, row-scaled B, FP32 out).
    * quantize with the transposed 128x1 output, X[16384,7168]; weight
      quantize W[7168,7168] with its transposed copy; power-of-two scale
      quantize and the FP8 re-tiling 1x128 -> 128x1 of the same X.
    """
    import torch
    out = {}
    reps = 10

    def gemm_line(flop, ms, **extra):
        tf = flop / (ms * 1e-3) / 1e12
        line = {"tflops": tf, "ms": ms, "frac_of_fp8_peak": tf / fp8_peak, "gflop": flop / 1e9, **extra}
        if hw_peak:
            line["frac_of_hw_rate"] = tf / hw_peak
        return line

    def bw_line(nbytes, ms, **extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"gbs": gbs, "ms": ms, "frac_of_hbm": gbs / hbm_peak, "frac_of_nominal_hbm": gbs / NOMINAL_HBM_GBS,
                "bytes": nbytes, **extra}

    if "dgrad" in sections:
        # ---- dgrad
        dy_bits, w_bits = synth.dgrad(seed=rank)
        dy = torch.from_numpy(dy_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        w = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        dyq, sdy = fp8bs.quantize_act(dy)
        _, _, wq_t, sw_t = fp8bs.quantize_weight(w, transposed=True)
        dx = torch.empty((4096, 2048), dtype=torch.float32, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_gemm(dyq, sdy, wq_t, sw_t, fp8bs.SCALE_BLOCK128x128, dx, fp8bs.OUT_F32,
                                               4096, 2048, 7168, 0, stream), stream, warmup, reps)
        out["dgrad"] = gemm_line(2.0 * 4096 * 2048 * 7168, ms, shape="M=4096 N=2048 K=7168, FP32 out")
        del dy, w, dyq, sdy, wq_t, sw_t, dx

    if "wgrad" in sections:
        # ---- wgrad (+ the dual-layout quantize of its operands)
        dy_bits, x_bits = synth.wgrad(seed=rank)
        dy = torch.from_numpy(dy_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        _, _, dyq_t, sdy_t = fp8bs.quantize_act(dy, transposed=True)
        xq, sx, xq_t, sx_t = fp8bs.quantize_act(x, transposed=True)
        dw = torch.empty((2048, 7168), dtype=torch.float32, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_gemm(dyq_t, sdy_t, xq_t, sx_t, fp8bs.SCALE_ROW1x128, dw, fp8bs.OUT_F32,
                                               2048, 7168, 16384, 0, stream), stream, warmup, reps)
        out["wgrad"] = gemm_line(2.0 * 2048 * 7168 * 16384, ms, shape="M=2048 N=7168 K=T=16384, row-scaled B, FP32 out")
        T_, K_ = x.shape
        ms = _time_ms(lambda: fp8bs.fp8bs_quantize_act(x, T_, K_, K_, xq, sx, xq_t, sx_t, stream), stream, warmup, reps)
        out["quantize_dual"] = bw_line(T_ * K_ * (2 + 1 + 1) + (T_ * (K_ // 128) + K_ * (T_ // 128)) * 4, ms,
                                       shape="X[16384,7168] -> 1x128 and 128x1")
        # power-of-two scales (§3.3.3 (1)) and the FP8 re-tiling 1x128 -> 128x1 (§3.5.2) of the same X
        ms = _time_ms(lambda: fp8bs.fp8bs_quantize_act_ex(x, T_, K_, K_, xq, sx, None, None, fp8bs.SCALE_POW2, stream),
                      stream, warmup, reps)
        out["quantize_pow2"] = bw_line(T_ * K_ * (2 + 1) + T_ * (K_ // 128) * 4, ms,
                                       shape="X[16384,7168] -> 1x128, power-of-two scales")
        ms = _time_ms(lambda: fp8bs.fp8bs_requant_1x128_to_128x1(xq, sx, T_, K_, xq_t, sx_t, fp8bs.SCALE_POW2, stream),
                      stream, warmup, reps)
        out["requant_1x128_to_128x1"] = bw_line(T_ * K_ * 2 + (T_ * (K_ // 128) + K_ * (T_ // 128)) * 4, ms,
                                                shape="X[16384,7168] FP8 1x128 -> 128x1 (dequantise, transpose, "
                                                      "requantise), power-of-two scales")
        del dy, x, dyq_t, sdy_t, xq, sx, xq_t, sx_t, dw

    if "context" in sections:
        # ---- context only (not part of the path): the library BF16 GEMM on the
        # dense fprop shape, to set the "FP8 ~ 2x BF16" claim of the pages beside
        # the block-scaled FP8 GEMM
        g0 = torch.Generator(device=dev)
        g0.manual_seed(2000 + rank)
        xa = torch.randn((4096, 7168), generator=g0, device=dev).to(torch.bfloat16)
        wa = (torch.randn((7168, 7168), generator=g0, device=dev) * 0.02).to(torch.bfloat16)
        ya = torch.empty((4096, 7168), dtype=torch.bfloat16, device=dev)
        ms = _time_ms(lambda: torch.matmul(xa, wa.t(), out=ya), stream, warmup, reps)
        out["context_bf16_matmul"] = gemm_line(2.0 * 4096 * 7168 * 7168, ms,
                                               shape="torch.matmul BF16 4096x7168x7168 (cuBLAS), context only")
        out["context_bf16_matmul"]["frac_of_bf16_peak"] = out["context_bf16_matmul"]["tflops"] / (fp8_peak / 2.0)
        del xa, wa, ya

    if "context" in sections:
        # ---- context only: accumulation precision without promotion.  The pages
        # (H800, all of K = 4096 accumulated in the tensor core) report a maximum
        # relative error near 2%; the diagnostic GEMM accumulates all of K in
        # tensor memory on this GPU, the production GEMM promotes every 128 K
        # (block scales 1 here).  Reference: the float64 product of the decoded
        # codes, exact for these sums (multiples of 2^-18 below 2^31).
        Mc, Nc, Kc = 128, 256, 4096
        ac = torch.randn((Mc, Kc), generator=g0, device=dev).to(torch.bfloat16)
        bc = torch.randn((Nc, Kc), generator=g0, device=dev).to(torch.bfloat16)
        acq, _ = fp8bs.quantize_act(ac, stream=stream)
        bcq, _ = fp8bs.quantize_act(bc, stream=stream)
        d_un = fp8bs.diag_gemm_unpromoted(acq, bcq, stream=stream)
        d_pr = fp8bs.gemm(acq, torch.ones((Kc // 128, Mc), device=dev), bcq,
                          torch.ones((Nc // 128, Kc // 128), device=dev), out_dtype=torch.float32, stream=stream)
        torch.cuda.synchronize(dev)
        yc = acq.view(torch.float8_e4m3fn).double() @ bcq.view(torch.float8_e4m3fn).double().t()
        big = yc.abs() >= 0.1 * yc.pow(2).mean().sqrt()

        def acc_err(d):
            e = (d.double() - yc).abs()
            return {"max_err_over_max_abs": float(e.max() / yc.abs().max()),
                    "max_rel_err": float((e[big] / yc[big].abs()).max())}

        out["context_unpromoted_accumulation"] = {
            "shape": f"{Mc}x{Nc}x{Kc}, E4M3 codes of N(0,1) in 1x128 groups, scales left out",
            "unpromoted_tensor_core": acc_err(d_un), "promoted_every_128": acc_err(d_pr),
            "pages_h800_unpromoted_max_rel_err": 0.02}
        del ac, bc, acq, bcq, d_un, d_pr, yc, big

    # one generator for the weight and MoE sections (the MoE weights follow W
    # in its stream when both run)
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    if "weight" in sections:
        # ---- weight quantize with the transposed copy
        wbig = (torch.randn((7168, 7168), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        wq, sw, wq_t2, sw_t2 = fp8bs.quantize_weight(wbig, transposed=True)
        ms = _time_ms(lambda: fp8bs.fp8bs_quantize_weight(wbig, 7168, 7168, 7168, wq, sw, wq_t2, sw_t2, stream),
                      stream, warmup, reps)
        out["quantize_weight"] = bw_line(7168 * 7168 * (2 + 1 + 1) + 2 * 56 * 56 * 4, ms,
                                         shape="W[7168,7168] -> 128x128 blocks + transposed copy")
        del wbig, wq, sw, wq_t2, sw_t2

    if "moe" in sections:
        # ---- MoE grouped fprop
        E, H, I = moe_experts, 7168, 2048
        choice = synth.moe_routing(seed=rank, tokens=moe_tokens, experts=E)
        offsets_np, src_np = synth.moe_layout(choice, E)
        rows = int(offsets_np[-1])
        real_rows = int((src_np >= 0).sum())
        x_tok = torch.from_numpy(synth.normal_bf16((moe_tokens, H), 1.0, rank, synth.TID_X,
                                                   outliers=True).view(np.int16))
        x_tok = x_tok.view(torch.bfloat16).to(dev)
        src = torch.from_numpy(src_np).to(dev)
        x_rows = torch.zeros((rows, H), dtype=torch.bfloat16, device=dev)
        ok = src >= 0
        x_rows[ok] = x_tok[src[ok]]
        offsets = torch.from_numpy(offsets_np).to(dev)
        w_gu = (torch.randn((E * 2 * I, H), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        w_dn = (torch.randn((E * H, I), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        d_in = torch.randn((rows, I), generator=g, device=dev).to(torch.bfloat16)
        d_in[~ok] = 0
        aq, sa = fp8bs.quantize_act(x_rows)
        bq, sb = fp8bs.quantize_weight(w_gu)
        y1 = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_grouped_gemm(aq, sa, rows, offsets, E, bq, sb, y1, fp8bs.OUT_BF16, 2 * I, H,
                                                       stream), stream, warmup, reps)
        out["moe_gate_up"] = gemm_line(2.0 * real_rows * 2 * I * H, ms, rows=rows, real_rows=real_rows,
                                       shape=f"grouped {E} experts, [{rows} x {2 * I} x {H}], BF16 out")
        # fused SwiGLU -> 1x128 quantise of the gate/up output (the down projection's input)
        sq = torch.empty((rows, I), dtype=torch.uint8, device=dev)
        ss = torch.empty((I // 128, rows), dtype=torch.float32, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_swiglu_quantize(y1, rows, I, 2 * I, sq, ss, fp8bs.SCALE_ABSMAX, stream),
                      stream, warmup, reps)
        out["swiglu_quantize"] = bw_line(rows * (2 * I * 2 + I + (I // 128) * 4), ms,
                                         shape=f"[{rows} x {2 * I}] BF16 gate|up -> SwiGLU -> 1x128 E4M3 [{rows} x {I}]")
        del aq, sa, bq, sb, y1, x_rows, w_gu, sq, ss
        aq, sa = fp8bs.quantize_act(d_in)
        bq, sb = fp8bs.quantize_weight(w_dn)
        y2 = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_grouped_gemm(aq, sa, rows, offsets, E, bq, sb, y2, fp8bs.OUT_BF16, H, I,
                                                       stream), stream, warmup, reps)
        out["moe_down"] = gemm_line(2.0 * real_rows * H * I, ms, rows=rows, real_rows=real_rows,
                                    shape=f"grouped {E} experts, [{rows} x {H} x {I}], BF16 out")
        del aq, sa, bq, sb, d_in, w_dn
        # ---- the data movement around the expert GEMMs on one rank (the
        # exchanges between ranks are the identity here): FP8 dispatch (pack:
        # scatter the tokens' codes with row-major scales to their send rows;
        # unpack: gather the received rows into the experts' padded segments
        # with kb-major scales; one rank: scatter straight into the segments)
        # and BF16 combine (the expert outputs back in send order, then the
        # gate-weighted sum; one rank: the sum reading the expert rows in place)
        from fp8_fine_grained_fp8bs_gb300 import moe as moe_plan
        plan = moe_plan.MoePlan(choice, E, 1)
        recv = moe_plan.exchange_counts(plan)
        R, T_, nkb = plan.T * plan.k, plan.T, H // 128
        xq_tok, sx_tok = fp8bs.quantize_act(x_tok, pow2=True)
        send_pos = torch.from_numpy(plan.send_pos).to(dev)
        unpack_idx = torch.from_numpy(recv.unpack_idx).to(dev)
        back_idx = torch.from_numpy(recv.back_idx).to(dev)
        local_pos = torch.from_numpy(recv.back_idx[plan.send_pos].astype(np.int32)).to(dev)
        pad_rows = torch.from_numpy(recv.pad_rows).to(dev)
        gate_w = torch.from_numpy(synth.moe_gate_weights(seed=rank, tokens=T_, top_k=plan.k)).to(dev)
        q_send = torch.empty((R, H), dtype=torch.uint8, device=dev)
        s_send = torch.empty((R, nkb), dtype=torch.float32, device=dev)
        q_exp = torch.empty((recv.padded_rows, H), dtype=torch.uint8, device=dev)
        s_exp = torch.empty((nkb, recv.padded_rows), dtype=torch.float32, device=dev)
        row_b = H + 4 * nkb
        # each token's row is read once and written to its k send positions
        ms = _time_ms(lambda: fp8bs.fp8bs_scatter_q_rows(xq_tok, sx_tok, T_, H, fp8bs.SCALES_KB_MAJOR, send_pos,
                                                         plan.k, None, 0, R, q_send, s_send, fp8bs.SCALES_ROW_MAJOR,
                                                         stream), stream, warmup, reps)
        out["moe_dispatch_pack"] = bw_line(T_ * row_b + R * row_b + 4 * R, ms,
                                           shape=f"{T_} tokens of E4M3 [{H}] + {nkb} scales scattered to their "
                                                 f"{R} (token, expert) send rows")
        ms = _time_ms(lambda: fp8bs.fp8bs_gather_q_rows(q_send, s_send, R, H, fp8bs.SCALES_ROW_MAJOR, unpack_idx,
                                                        recv.padded_rows, q_exp, s_exp, fp8bs.SCALES_KB_MAJOR, stream),
                      stream, warmup, reps)
        out["moe_dispatch_unpack"] = bw_line(R * row_b + recv.padded_rows * (row_b + 4), ms,
                                             shape=f"{R} received rows into {E} expert segments padded to 128 "
                                                   f"({recv.padded_rows} rows)")
        n_pad = int(recv.pad_rows.size)
        ms = _time_ms(lambda: fp8bs.fp8bs_scatter_q_rows(xq_tok, sx_tok, T_, H, fp8bs.SCALES_KB_MAJOR, local_pos,
                                                         plan.k, pad_rows, n_pad, recv.padded_rows, q_exp, s_exp,
                                                         fp8bs.SCALES_KB_MAJOR, stream), stream, warmup, reps)
        out["moe_dispatch_local"] = bw_line(T_ * row_b + recv.padded_rows * row_b + 4 * (R + n_pad), ms,
                                            shape=f"one rank: {T_} tokens scattered straight into {E} expert "
                                                  f"segments padded to 128 ({recv.padded_rows} rows, {n_pad} "
                                                  f"zeroed)")
        y_back = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
        comb = torch.empty((T_, H), dtype=torch.bfloat16, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_gather_bf16_rows(y2, rows, H, back_idx, R, y_back, stream), stream, warmup,
                      reps)
        out["moe_combine_gather"] = bw_line(2 * R * H * 2 + 4 * R, ms,
                                            shape=f"{R} BF16 expert output rows [{H}] back in send order")
        ms = _time_ms(lambda: fp8bs.fp8bs_moe_combine(y_back, R, H, send_pos, gate_w, T_, plan.k, comb, stream), stream,
                      warmup, reps)
        out["moe_combine"] = bw_line(R * H * 2 + T_ * H * 2 + 8 * R, ms,
                                     shape=f"{T_} tokens x top-{plan.k}: gate-weighted BF16 sum in FP32 -> BF16 [{H}]")
        ms = _time_ms(lambda: fp8bs.fp8bs_moe_combine(y2, rows, H, local_pos, gate_w, T_, plan.k, comb, stream),
                      stream, warmup, reps)
        out["moe_combine_local"] = bw_line(R * H * 2 + T_ * H * 2 + 8 * R, ms,
                                           shape="one rank: the same sum reading the expert rows in place")
        # ---- the whole MoE layer on one rank, launched back to back as a user
        # runs it: FP8 dispatch (scatter into the padded expert segments), the
        # gate/up grouped GEMM, the fused SwiGLU quantise, the down grouped GEMM
        # and the BF16 combine; TFLOP/s of the two GEMMs' real-row flops
        del y_back
        w_gu = (torch.randn((E * 2 * I, H), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        gq, gs = fp8bs.quantize_weight(w_gu)
        del w_gu
        w_dn = (torch.randn((E * H, I), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        dq, ds = fp8bs.quantize_weight(w_dn)
        del w_dn
        gq, gs = gq.view(E, 2 * I, H), gs.view(E, 2 * I // 128, H // 128)
        dq, ds = dq.view(E, H, I), ds.view(E, H // 128, I // 128)
        seg = torch.from_numpy(recv.offsets).to(dev)
        h1 = torch.empty((recv.padded_rows, 2 * I), dtype=torch.bfloat16, device=dev)
        hq = torch.empty((recv.padded_rows, I), dtype=torch.uint8, device=dev)
        hs = torch.empty((I // 128, recv.padded_rows), dtype=torch.float32, device=dev)

        def moe_layer():
            fp8bs.fp8bs_scatter_q_rows(xq_tok, sx_tok, T_, H, fp8bs.SCALES_KB_MAJOR, local_pos, plan.k, pad_rows,
                                       n_pad, recv.padded_rows, q_exp, s_exp, fp8bs.SCALES_KB_MAJOR, stream)
            fp8bs.fp8bs_grouped_gemm(q_exp, s_exp, recv.padded_rows, seg, E, gq, gs, h1, fp8bs.OUT_BF16, 2 * I, H,
                                     stream)
            fp8bs.fp8bs_swiglu_quantize(h1, recv.padded_rows, I, 2 * I, hq, hs, fp8bs.SCALE_ABSMAX, stream)
            fp8bs.fp8bs_grouped_gemm(hq, hs, recv.padded_rows, seg, E, dq, ds, y2, fp8bs.OUT_BF16, H, I, stream)
            fp8bs.fp8bs_moe_combine(y2, recv.padded_rows, H, local_pos, gate_w, T_, plan.k, comb, stream)

        ms = _time_ms(moe_layer, stream, warmup, reps)
        if fp8bs.fp8bs_get_device_status(stream) != 0:
            raise RuntimeError("device status after the MoE layer")
        out["moe_layer"] = gemm_line(2.0 * R * (2 * I * H + H * I), ms, rows=recv.padded_rows, real_rows=R,
                                     shape=f"one rank, {T_} tokens x top-{plan.k} of {E} experts, hidden {H}, "
                                           f"expert {I}: dispatch, gate/up GEMM, SwiGLU quantise, down GEMM, "
                                           "combine (5 launches)")
        out["moe_layer"]["launches"] = 5
        del y2, xq_tok, sx_tok, q_send, s_send, q_exp, s_exp, comb, local_pos, pad_rows, gq, gs, dq, ds, h1, hq, hs
    if "pow2" in sections:
        # ---- power-of-two scales applied by the tensor core (UE8M0 block
        # scales of tcgen05.mma.kind::mxf8f6f4), next to the fold GEMM on the
        # same operands: the dense fprop shape, the MoE expert GEMMs and Wgrad
        x_bits, w_bits = synth.dense_fprop(seed=rank)
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        w = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        xq, sx = fp8bs.quantize_act(x, pow2=True)
        wq, sw = fp8bs.quantize_weight(w, pow2=True)
        yp = torch.empty((4096, 7168), dtype=torch.bfloat16, device=dev)
        flop = 2.0 * 4096 * 7168 * 7168
        ms = _time_ms(lambda: fp8bs.fp8bs_gemm_pow2(xq, sx, wq, sw, fp8bs.SCALE_BLOCK128x128, yp, fp8bs.OUT_BF16,
                                                    4096, 7168, 7168, 0, stream), stream, warmup, reps)
        out["gemm_pow2_dense"] = gemm_line(flop, ms, shape="M=4096 N=7168 K=7168, power-of-two scales in the MMA "
                                                            "(kind::mxf8f6f4, UE8M0), BF16 out")
        ms = _time_ms(lambda: fp8bs.fp8bs_gemm(xq, sx, wq, sw, fp8bs.SCALE_BLOCK128x128, yp, fp8bs.OUT_BF16,
                                               4096, 7168, 7168, 0, stream), stream, warmup, reps)
        out["gemm_fold_dense_same_operands"] = gemm_line(flop, ms, shape="the same power-of-two operands through "
                                                                         "the CUDA-core fold GEMM")
        del x, w, xq, sx, wq, sw, yp
        # Wgrad: dY re-tiled 1x128 -> 128x1 from FP8 (power-of-two), X quantised 128x1
        dy_bits, x_bits = synth.wgrad(seed=rank)
        dy = torch.from_numpy(dy_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        dyq, sdy = fp8bs.quantize_act(dy, pow2=True)
        dyq_t, sdy_t = fp8bs.requant_1x128_to_128x1(dyq, sdy, pow2=True)
        _, _, xq_t, sx_t = fp8bs.quantize_act(x, transposed=True, pow2=True)
        dw = torch.empty((2048, 7168), dtype=torch.float32, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_gemm_pow2(dyq_t, sdy_t, xq_t, sx_t, fp8bs.SCALE_ROW1x128, dw,
                                                    fp8bs.OUT_F32, 2048, 7168, 16384, 0, stream), stream, warmup, reps)
        out["wgrad_pow2"] = gemm_line(2.0 * 2048 * 7168 * 16384, ms,
                                      shape="M=2048 N=7168 K=T=16384, row-scaled B, power-of-two scales in the MMA, "
                                            "FP32 out")
        del dy, x, dyq, sdy, dyq_t, sdy_t, xq_t, sx_t, dw
        # MoE expert GEMMs with power-of-two activation and weight scales
        E, H, I = moe_experts, 7168, 2048
        choice = synth.moe_routing(seed=rank, tokens=moe_tokens, experts=E)
        offsets_np, src_np = synth.moe_layout(choice, E)
        rows = int(offsets_np[-1])
        real_rows = int((src_np >= 0).sum())
        offsets = torch.from_numpy(offsets_np).to(dev)
        gp = torch.Generator(device=dev)
        gp.manual_seed(3000 + rank)
        ok = torch.from_numpy(src_np).to(dev) >= 0
        a_in = torch.randn((rows, H), generator=gp, device=dev).to(torch.bfloat16)
        a_in[~ok] = 0
        w_gu = (torch.randn((E * 2 * I, H), generator=gp, device=dev) * 0.02).to(torch.bfloat16)
        aq, sa = fp8bs.quantize_act(a_in, pow2=True)
        bq, sb = fp8bs.quantize_weight(w_gu, pow2=True)
        y1 = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_grouped_gemm_pow2(aq, sa, rows, offsets, E, bq, sb, y1, fp8bs.OUT_BF16,
                                                            2 * I, H, stream), stream, warmup, reps)
        out["moe_gate_up_pow2"] = gemm_line(2.0 * real_rows * 2 * I * H, ms, rows=rows, real_rows=real_rows,
                                            shape=f"grouped {E} experts, [{rows} x {2 * I} x {H}], power-of-two "
                                                  f"scales in the MMA, BF16 out")
        del a_in, w_gu, aq, sa, bq, sb, y1
        d_in = torch.randn((rows, I), generator=gp, device=dev).to(torch.bfloat16)
        d_in[~ok] = 0
        w_dn = (torch.randn((E * H, I), generator=gp, device=dev) * 0.02).to(torch.bfloat16)
        aq, sa = fp8bs.quantize_act(d_in, pow2=True)
        bq, sb = fp8bs.quantize_weight(w_dn, pow2=True)
        y2 = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
        ms = _time_ms(lambda: fp8bs.fp8bs_grouped_gemm_pow2(aq, sa, rows, offsets, E, bq, sb, y2, fp8bs.OUT_BF16,
                                                            H, I, stream), stream, warmup, reps)
        out["moe_down_pow2"] = gemm_line(2.0 * real_rows * H * I, ms, rows=rows, real_rows=real_rows,
                                         shape=f"grouped {E} experts, [{rows} x {H} x {I}], power-of-two scales in "
                                               f"the MMA, BF16 out")
        del d_in, w_dn, aq, sa, bq, sb, y2, ok
    if fp8bs.fp8bs_get_device_status(stream) != 0:
        raise RuntimeError("device status after the workload measurements")
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="fp8bs", choices=["fp8bs", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-kernel lines of the MoE, dgrad, wgrad and quantize variants")
    ap.add_argument("--workloads", default=",".join(WORKLOAD_SECTIONS),
                    help="comma-separated sections of the per-kernel lines to run: " + ", ".join(WORKLOAD_SECTIONS)
                         + " (wgrad also times the dual, power-of-two and re-tiling quantisations of its X; "
                           "moe the grouped GEMMs and the fused SwiGLU quantisation)")
    ap.add_argument("--moe-tokens", type=int, default=8192,
                    help="tokens of the MoE workload (8192: the benchmark's; smaller for profiling captures)")
    ap.add_argument("--moe-experts", type=int, default=32,
                    help="experts of the MoE workload (32: the benchmark's; top-8 routing needs at least 8)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.sections = tuple(w for w in args.workloads.split(",") if w)
    unknown = set(args.sections) - set(WORKLOAD_SECTIONS)
    if unknown:
        ap.error(f"unknown workload sections: {sorted(unknown)}")
    if args.moe_experts < 8 or args.moe_tokens < 1:
        ap.error("--moe-experts must be at least 8 (top-8 routing) and --moe-tokens positive")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import fp8_fine_grained_fp8bs_gb300 as fp8bs
    from fp8_fine_grained_fp8bs_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v: float) -> float:
        if world == 1:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    fp8bs.build()
    fp8bs.load_library()
    stream = torch.cuda.current_stream(dev)

    # inputs: each rank its own batch (replica), resident in HBM before timing
    x_bits, w_bits = synth.dense_fprop(seed=rank)
    xin = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    win = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    wq = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    # X (1x128) and W (128x128) are quantised by one launch whose persistent
    # grid walks X's tiles, then W's; then the GEMM.
    def quantize_step():
        fp8bs.fp8bs_quantize_act_weight(xin, M, K, K, xq, sx, win, N, K, K, wq, sw, fp8bs.SCALE_ABSMAX, stream)

    def gemm_step():
        fp8bs.fp8bs_gemm(xq, sx, wq, sw, fp8bs.SCALE_BLOCK128x128, y, fp8bs.OUT_BF16, M, N, K, 0, stream)

    for _ in range(args.warmup):
        quantize_step()
        gemm_step()
    torch.cuda.synchronize(dev)
    if fp8bs.fp8bs_get_device_status(stream) != 0:
        raise RuntimeError("device status after warm-up")

    # the steps: nothing recorded between the two launches of a step
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(_gpu_id(torch, local))
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for _ in range(args.steps):
        quantize_step()
        gemm_step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    ms_step = max_over_ranks(t_start.elapsed_time(t_end) / args.steps)
    if fp8bs.fp8bs_get_device_status(stream) != 0:
        raise RuntimeError("device status after the timed steps")

    # the GEMM alone, in steps of a pass of its own: the quantisation runs
    # before each GEMM as in the step (its 161 MB read leaves in L2 only what
    # it wrote, the GEMM's operands), CUDA events around the GEMM launch alone
    # on the launching stream (the dominant kernel's roofline); nothing is
    # recorded between the launches of the timed steps above
    ng = max(10, min(args.steps, 200))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ng)]
    barrier()
    torch.cuda.synchronize(dev)
    for a, b in ev:
        quantize_step()
        a.record(stream)
        gemm_step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    gemm_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev))

    # standalone quantize of X[16384, 7168] (inputs 235 MB > L2)
    xl_bits = synth.quantize_input(seed=rank)
    xl = torch.from_numpy(xl_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    xlq = torch.empty((QM, QK), dtype=torch.uint8, device=dev)
    xls = torch.empty((QK // 128, QM), dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        fp8bs.fp8bs_quantize_act(xl, QM, QK, QK, xlq, xls, None, None, stream)
    nq = max(10, min(args.steps, 200))
    qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nq)]
    barrier()
    torch.cuda.synchronize(dev)
    for a, b in qev:
        a.record(stream)
        fp8bs.fp8bs_quantize_act(xl, QM, QK, QK, xlq, xls, None, None, stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    q_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in qev))
    del xl, xlq, xls

    # End to end through the public API with host buffers: every step copies
    # its X and W from pinned host memory and reads its Y back.  The steps are
    # pipelined over three streams (copy in, compute, copy out) with double
    # device buffers, so step i+1's inputs travel while step i computes.
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    w_host = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    ne = max(4, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    xb = [xin, torch.empty_like(xin)]
    wb = [win, torch.empty_like(win)]
    yb = [y, torch.empty_like(y)]
    xqb = [xq, torch.empty_like(xq)]
    sxb = [sx, torch.empty_like(sx)]
    wqb = [wq, torch.empty_like(wq)]
    swb = [sw, torch.empty_like(sw)]

    def e2e_run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            j = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])          # buffers j free again
                xb[j].copy_(x_host, non_blocking=True)
                wb[j].copy_(w_host, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])             # yb[j] read out
            fp8bs.fp8bs_quantize_act_weight(xb[j], M, K, K, xqb[j], sxb[j], wb[j], N, K, K, wqb[j], swb[j],
                                            fp8bs.SCALE_ABSMAX, stream)
            fp8bs.fp8bs_gemm(xqb[j], sxb[j], wqb[j], swb[j], fp8bs.SCALE_BLOCK128x128, yb[j], fp8bs.OUT_BF16,
                             M, N, K, 0, stream)
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                y_host.copy_(yb[j], non_blocking=True)
                ev_out[i].record(s_out)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    e2e_run(3)
    barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    e2e_run(ne)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / ne)
    if fp8bs.fp8bs_get_device_status(stream) != 0:
        raise RuntimeError("device status after the end-to-end steps")

    peaks, peak_src = _peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = peaks.get("sm_max_mhz") or clocks.get("sm_max_mhz") or 2070.0
    hw_peak = hw_fp8_peak_tflops(sms, max_mhz)
    workloads = None
    if not args.no_workloads:
        workloads = measure_workloads(fp8bs, synth, dev, stream, rank, fp8_peak, peaks["hbm_gbs"], args.warmup,
                                      args.sections, args.moe_tokens, args.moe_experts, hw_peak)
    gemm_tflops = GEMM_FLOP / (gemm_ms * 1e-3) / 1e12
    q_gbs = QUANT_BYTES / (q_ms * 1e-3) / 1e9
    value = world * GEMM_FLOP / (ms_step * 1e-3) / 1e12
    # The contract keys first, then the per-configuration lines, and the
    # dominant kernels' figures last (the end of the line is what a truncated
    # log keeps).
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "out": "bf16",
                   "quantize_shape": [QM, QK], "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (X+W BF16 = 161 MB per step > 129 MB), no flush; the GEMM "
                         "alone is timed in a pass of its own with the quantisation before each launch, as in "
                         "the step"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": {"value": world * GEMM_FLOP / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(xin.numel() * 2 + win.numel() * 2),
                "d2h_bytes_per_step": int(y.numel() * 2), "ms_per_step": e2e_ms},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x_bits, w_bits, xl_bits)
    if workloads is not None:
        line["workloads"] = workloads
    line["roofline"] = {
        "bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
        "frac": gemm_tflops / fp8_peak,
        "traffic": _traffic("gemm_dense_fprop_bf16", *(CSRC + f for f in ("gemm.cu", "gemm_common.cuh", "common.cuh"))),
        "peak_source": f"{peak_src}: bf16 burst x {FP8_OVER_BF16:g} (nominal FP8/BF16)",
        "hw_rate_peak": hw_peak, "frac_of_hw_rate": gemm_tflops / hw_peak,
        "hw_rate_source": f"{sms} SMs x 16384 FP8 FLOP/clk/SM x {max_mhz:g} MHz (maximum SM clock)"}
    if clocks.get("sm_mhz"):
        hw_med = hw_fp8_peak_tflops(sms, clocks["sm_mhz"])
        line["roofline"]["hw_rate_peak_median_clock"] = hw_med
        line["roofline"]["frac_of_hw_rate_median_clock"] = gemm_tflops / hw_med
    line["gemm"] = {"tflops": gemm_tflops, "ms": gemm_ms, "frac_of_fp8_peak": gemm_tflops / fp8_peak,
                    "frac_of_hw_rate": gemm_tflops / hw_peak}
    line["quantize_roofline"] = {
        "bound": "hbm", "achieved": q_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": q_gbs / peaks["hbm_gbs"],
        "traffic": _traffic("quantize_act_1x128_16384x7168", *(CSRC + f for f in ("quantize.cu", "common.cuh"))),
        "peak_source": peak_src, "frac_of_nominal_hbm": q_gbs / NOMINAL_HBM_GBS,
        "nominal_hbm_gbs": NOMINAL_HBM_GBS}
    line["quantize"] = {"gbs": q_gbs, "ms": q_ms, "frac_of_hbm": q_gbs / peaks["hbm_gbs"],
                        "frac_of_nominal_hbm": q_gbs / NOMINAL_HBM_GBS, "bytes": QUANT_BYTES}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
