"""Benchmark of the fused MaxSim hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One *step* is one fused forward (scores + the saved argmax) of 16 queries
(Lq = 32) against a 50,000-document ColBERT-shaped corpus with Ld uniform in
[32, 300], packed with cu_seqlens, FP16 (the padding-free rerank of
"FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval",
§4.3.2).  The metric is documents scored per second (each document against
all 16 queries).  Inputs are seeded synthetic unit-norm embeddings (no
dataset is read) and exceed L2 (2.1 GB of documents vs a 129 MB L2), so
every step streams them from HBM.

Under torchrun (N > 1) every rank scores its own 50,000-document shard (weak
scaling; no collective on the data path, only the timing barrier and max).

Rank 0 prints ONE JSON line.  Besides the contract keys it carries:
  roofline      the forward kernel's achieved tensor throughput (algorithmic
                FLOPs / its CUDA-event duration) against the measured peak,
  cpu_baseline  the CPU oracle timed on the host cores on a bounded sample,
  e2e           the same metric with host-resident inputs copied in and the
                scores copied back every step,
  clocks        SM clocks sampled by nvidia-smi during the timed region,
  extra         the other workloads (ColPali, training fwd+bwd, INT8 with one
                scale per tensor and per token, the two-stage INT8 -> FP16
                top-K scan, out-of-core scoring of a host-resident corpus,
                and the Chamfer distance of two 100K-point clouds).

``--impl reference`` times the CPU oracle (the only reference this method
has) on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "docs scored/s"
UNIT = "docs/s"
WORKLOAD = "colbert_varlen"
L2_BYTES = 129 * 2**20


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, when it was taken
    on the current kernel sources (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(workload)
    if not rec:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return rec["dram_bytes_per_launch"] if rec.get("source_sha256_16") == h.hexdigest()[:16] else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (background)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- multi-rank

def rank_workload(w, rank: int):
    """Weak scaling: every rank scores its own shard of the same shape, drawn
    with a rank-specific seed (documents never move between ranks)."""
    from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
    return syn.Workload(w.name, w.n_q, w.lq, w.n_docs, w.ld_lo, w.ld_hi, w.dtype, seed=w.seed + rank)


def max_over_ranks(value: float, device) -> float:
    """The slowest rank's time (the job finishes when it does); the only
    collective of the benchmark, outside the timed region's data path."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------- ours

def _time_loop(fn, steps, warmup, stream, nvtx=None):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if nvtx:
        torch.cuda.nvtx.range_push(nvtx)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s, e in ev:
        s.record(stream)
        fn()
        e.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if nvtx:
        torch.cuda.nvtx.range_pop()
    per = [s.elapsed_time(e) for s, e in ev]
    return t0.elapsed_time(t1), per


def _forward_launches(lq_max: int, int8: bool) -> int:
    lq_pad = 1 << max(0, (lq_max - 1).bit_length()) if lq_max <= 32 else -(-lq_max // 32) * 32
    return 1 + (1 if lq_pad > 32 else 0) + (1 if int8 else 0)


def _l2_read_gbs(m, mib=48, passes=20):
    """The SMs' read rate from L2: the library's plain-read probe over a
    48 MiB buffer (L2-resident: the L2 holds 129 MB), one warm pass, then
    `passes` timed passes (median of 5 launches)."""
    import torch
    stream = torch.cuda.current_stream()
    buf = torch.zeros(mib << 20, dtype=torch.uint8, device="cuda")
    sink = m.maxsim_probe_l2_read(buf, 1)
    _, per = _time_loop(lambda: m.maxsim_probe_l2_read(buf, passes, sink=sink), 5, 2, stream)
    gbs = buf.numel() * passes / (statistics.median(per) / 1e3) / 1e9
    del buf, sink
    return gbs


def _extra_workloads(m, syn, rl, peaks):
    """Shorter timings of the other workloads: forwards as the median of 50
    CUDA-event reps after 10 warm-up calls (p10 / p90 beside it), the rest of
    20."""
    import torch
    out = {}
    stream = torch.cuda.current_stream()
    l2_gbs = _l2_read_gbs(m)
    out["l2_read_gbs"] = round(l2_gbs, 1)
    for name in ("colbert_varlen", "colbert_1q", "colpali", "train", "train_colpali", "int8_varlen"):
        w = syn.WORKLOADS[name]
        torch.cuda.empty_cache()
        base_bytes = torch.cuda.memory_allocated()   # what earlier lines still hold
        x = syn.make_inputs(w, device="cuda")
        torch.cuda.reset_peak_memory_stats()         # not the generator's temporaries
        Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
        kw = dict(q_scale=x["q_scale"], d_scale=x["d_scale"])
        s, a, _ = m.maxsim_forward(Q, ql, D, cu, **kw)
        ws = torch.empty(max(1, m.maxsim_forward_workspace_size(w.n_q, w.lq, w.n_docs, w.dtype)),
                         dtype=torch.uint8, device="cuda")
        _, per = _time_loop(lambda: m.maxsim_forward(Q, ql, D, cu, scores=s, argmax=a, workspace=ws,
                                                     **kw), 50, 10, stream)
        ms = statistics.median(per)
        dec = statistics.quantiles(per, n=10)   # deciles: p10 .. p90
        # device memory held by one forward: inputs, outputs and workspace
        # (the similarity tensor is never materialised; its FP32 size for
        # comparison)
        peak_bytes = torch.cuda.max_memory_allocated() - base_bytes
        _, per_v = _time_loop(lambda: m.maxsim_forward(Q, ql, D, cu, with_argmax=False, scores=s, workspace=ws,
                                                       **kw), 20, 3, stream)
        flops = rl.forward_flops(int(ql.sum()), D.shape[0])
        rec = {"n_q": w.n_q, "lq": w.lq, "n_docs": w.n_docs, "ld": [w.ld_lo, w.ld_hi],
               "dtype": w.dtype, "fwd_ms": round(ms, 4), "fwd_p10_ms": round(dec[0], 4),
               "fwd_p90_ms": round(dec[-1], 4), "docs_per_s": w.n_docs / (ms / 1e3),
               # query-token x document-token similarities formed (and folded) per second
               "token_pairs_per_s": int(ql.sum()) * D.shape[0] / (ms / 1e3),
               "fwd_tflops": flops / (ms / 1e3) / 1e12,
               "fwd_frac_of_measured_bf16_peak": flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
               "fwd_value_only_ms": round(statistics.median(per_v), 4),
               "peak_device_bytes": int(peak_bytes),
               "similarity_tensor_fp32_bytes": int(ql.sum()) * D.shape[0] * 4}
        if name == "colbert_1q":
            # one query: 32 FLOP per document byte, far below the ridge -- HBM-bound
            hb = rl.forward_hbm_bytes(w.n_q, w.lq, w.n_docs, D.shape[0])
            rec["roofline"] = {"bound": "hbm", "achieved": round(hb / (ms / 1e3) / 1e9, 1),
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": round(hb / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 3),
                               "algorithmic_bytes_per_launch": hb}
        if name.startswith("train"):
            n = s.shape[0]
            g = torch.softmax(s / 0.05, dim=1)
            g[torch.arange(n), torch.arange(n)] -= 1.0
            g = g.contiguous()
            bws = torch.empty(m.maxsim_backward_workspace_size(w.n_q, w.lq, w.n_docs, D.shape[0]),
                              dtype=torch.uint8, device="cuda")
            dq, dd = m.maxsim_backward(g, a, Q, ql, D, cu, workspace=bws)
            _, perb = _time_loop(lambda: m.maxsim_backward(g, a, Q, ql, D, cu, dQ=dq, dD=dd,
                                                           workspace=bws), 50, 10, stream)
            msb = statistics.median(perb)
            decb = statistics.quantiles(perb, n=10)

            # one training step, forward then backward, on resident inputs
            def train_step():
                m.maxsim_forward(Q, ql, D, cu, scores=s, argmax=a, workspace=ws)
                m.maxsim_backward(g, a, Q, ql, D, cu, dQ=dq, dD=dd, workspace=bws)
            _, pers = _time_loop(train_step, 20, 3, stream)
            # and end to end through the C ABI with host buffers: Q and D in,
            # forward, the upstream gradient (here the synthetic contrastive
            # one, computed from the scores on the device), backward, dQ and
            # dD out
            Qh, Dh = Q.cpu().pin_memory(), D.cpu().pin_memory()
            dqh = torch.empty(dq.shape, dtype=torch.float32).pin_memory()
            ddh = torch.empty(dd.shape, dtype=torch.float32).pin_memory()

            def train_e2e():
                Q.copy_(Qh, non_blocking=True)
                D.copy_(Dh, non_blocking=True)
                m.maxsim_forward(Q, ql, D, cu, scores=s, argmax=a, workspace=ws)
                ge = torch.softmax(s / 0.05, dim=1)
                ge[torch.arange(n, device="cuda"), torch.arange(n, device="cuda")] -= 1.0
                m.maxsim_backward(ge, a, Q, ql, D, cu, dQ=dq, dD=dd, workspace=bws)
                dqh.copy_(dq, non_blocking=True)
                ddh.copy_(dd, non_blocking=True)
            _, pere = _time_loop(train_e2e, 10, 3, stream)
            rec.update(train_step_ms=round(statistics.median(pers), 4),
                       train_step_e2e_ms=round(statistics.median(pere), 4),
                       train_e2e_h2d_bytes=Qh.numel() * Qh.element_size() + Dh.numel() * Dh.element_size(),
                       train_e2e_d2h_bytes=dqh.numel() * 4 + ddh.numel() * 4)
            del Qh, Dh, dqh, ddh
            bb = rl.backward_hbm_bytes(w.n_q, w.lq, w.n_docs, D.shape[0], int(ql.sum()) * w.n_docs)
            n_src = int(ql.sum()) * w.n_docs
            gather = 2 * n_src * w.dim * 2
            rec.update(bwd_ms=round(msb, 4), bwd_p10_ms=round(decb[0], 4), bwd_p90_ms=round(decb[-1], 4),
                       step_ms=round(ms + msb, 4),
                       bwd_algorithmic_bytes=bb["total"],
                       bwd_l2_gather_bytes=gather,
                       bwd_gbs=bb["total"] / (msb / 1e3) / 1e9,
                       bwd_frac_of_measured_hbm=bb["total"] / (msb / 1e3) / 1e9 / peaks["hbm_gbs"],
                       # the gathers read 256-byte rows of an L2-resident Q / D: the
                       # bound is the SMs' L2 read rate (measured above by the probe)
                       bwd_roofline={"bound": "l2", "achieved": round((gather + bb["total"]) / (msb / 1e3) / 1e9, 1),
                                     "peak": round(l2_gbs, 1), "unit": "GB/s",
                                     "frac": round((gather + bb["total"]) / (msb / 1e3) / 1e9 / l2_gbs, 3),
                                     "bytes": gather + bb["total"],
                                     "peak_source": "maxsim_probe_l2_read, 48 MiB buffer, this run"})
        if m.maxsim_device_status() != 0:
            rec["device_status"] = "fault"
        out[name] = rec
        del x, Q, D, s, a
        ws = cu = ql = g = bws = dq = dd = None
        torch.cuda.empty_cache()
    out["out_of_core_colpali"] = _out_of_core(m, syn)
    out.update(_int8_variants(m, syn))
    return out


def _out_of_core(m, syn, steps=3, n_docs=100_000, block_docs=20_000, ld=1024, lq=1024):
    """Flash-MaxSim §5 "Out-of-Core Corpus Scaling": one ColPali query
    (Lq = Ld = 1024, FP16) against a corpus held in pinned host memory and
    streamed to the device in blocks of 20,000 documents.  The bound is the
    host-to-device link, so the roofline denominator is a plain pinned copy
    measured here; the device footprint is the two staging blocks."""
    import torch
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    total = n_docs * ld
    D_h = torch.empty((total, 128), dtype=torch.float16, pin_memory=True)
    chunk = 10_000
    for c in range(0, n_docs, chunk):
        k = min(chunk, n_docs - c)
        D_h[c * ld:(c + k) * ld].copy_(syn.unit_tokens(k * ld, 128, 1000 + c, "fp16", dev))
    cu_h = torch.arange(0, total + 1, ld, dtype=torch.int32).pin_memory()
    Q = syn.unit_tokens(lq, 128, 7, "fp16", dev).view(1, lq, 128)
    ql = torch.tensor([lq], dtype=torch.int32, device=dev)
    scores = torch.empty((1, n_docs), dtype=torch.float32, device=dev)
    ws = torch.empty(m.maxsim_forward_host_workspace_size(1, lq, n_docs, block_docs, block_docs * ld, "fp16"),
                     dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def call():
        m.maxsim_forward_host(Q, ql, D_h, cu_h, block_docs=block_docs, block_tokens=block_docs * ld,
                              scores=scores, workspace=ws)
    # the link's own rate: each block's bytes, pinned host -> device, plain
    # copies, taken before and after the timed calls; the best block is the
    # denominator (the host memory is shared with other jobs, so a single
    # copy can read far below the link)
    def link_rate():
        best = 0.0
        for b0 in range(0, n_docs, block_docs):
            blk = D_h[b0 * ld:(b0 + block_docs) * ld]
            dst = ws[: blk.numel() * 2].view(torch.float16).view(-1, 128)
            _, cp = _time_loop(lambda: dst.copy_(blk, non_blocking=True), 2, 1, stream)
            best = max(best, blk.numel() * 2 / (min(cp) / 1e3) / 1e9)
        return best
    link_before = link_rate()
    _, per = _time_loop(call, steps, 1, stream)
    ms = statistics.median(per)
    link_gbs = max(link_before, link_rate())
    corpus_bytes = total * 128 * 2
    achieved = corpus_bytes / (ms / 1e3) / 1e9
    rec = {"n_q": 1, "lq": lq, "n_docs": n_docs, "ld": ld, "dtype": "fp16", "block_docs": block_docs,
           "corpus_bytes_host": corpus_bytes, "call_ms": round(ms, 2), "docs_per_s": n_docs / (ms / 1e3),
           "host_link_gbs": round(achieved, 1), "measured_pinned_copy_gbs": round(link_gbs, 1),
           "frac_of_measured_copy": round(achieved / link_gbs, 3),
           "device_bytes": ws.numel() + Q.numel() * 2 + scores.numel() * 4 + 4}
    if m.maxsim_device_status() != 0:
        rec["device_status"] = "fault"
    del D_h, cu_h, ws
    torch.cuda.empty_cache()
    return rec


def _int8_variants(m, syn, steps=10):
    """§4.3.1 per-token INT8 on the 32 x 32 vs 100,000-document varlen shape,
    and the two-stage INT8 -> FP16 top-K scan (§4.1 "Kernel Family") on the
    same corpus: INT8 scan of every document, 1,000 candidates per query
    rescored in FP16, the best 100 returned."""
    import torch
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    w = syn.WORKLOADS["int8_varlen"]
    cu = syn.cu_seqlens_from_lengths(syn.doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed)).to(dev)
    total = int(cu[-1])
    ql = torch.full((w.n_q,), w.lq, dtype=torch.int32, device=dev)
    out = {}
    Q8, qs = syn.unit_tokens_int8_per_token(w.n_q * w.lq, w.dim, w.seed + 1, dev)
    D8, ds = syn.unit_tokens_int8_per_token(total, w.dim, w.seed + 2, dev)
    Q8, qs = Q8.view(w.n_q, w.lq, w.dim), qs.view(w.n_q, w.lq)
    s, a = m.maxsim_forward_int8_per_token(Q8, qs, ql, D8, ds, cu)
    _, per = _time_loop(lambda: m.maxsim_forward_int8_per_token(Q8, qs, ql, D8, ds, cu, scores=s, argmax=a),
                        steps, 3, stream)
    ms = statistics.median(per)
    out["int8_per_token"] = {"n_q": w.n_q, "lq": w.lq, "n_docs": w.n_docs, "ld": [w.ld_lo, w.ld_hi],
                             "fwd_ms": round(ms, 4), "docs_per_s": w.n_docs / (ms / 1e3)}
    del Q8, D8, qs, ds, s, a
    Q8, qst = syn.unit_tokens_int8(w.n_q * w.lq, w.dim, w.seed + 1, dev)
    D8, dst = syn.unit_tokens_int8(total, w.dim, w.seed + 2, dev)
    Q8 = Q8.view(w.n_q, w.lq, w.dim)
    Q16 = syn.unit_tokens(w.n_q * w.lq, w.dim, w.seed + 1, "fp16", dev).view(w.n_q, w.lq, w.dim)
    D16 = syn.unit_tokens(total, w.dim, w.seed + 2, "fp16", dev)
    kc, k = 1000, 100
    ws = torch.empty(m.maxsim_rerank_workspace_size(w.n_q, w.lq, w.n_docs, kc, w.ld_hi, "fp16"),
                     dtype=torch.uint8, device=dev)

    def rerank():
        m.maxsim_rerank_two_stage(Q8, D8, Q16, D16, ql, cu, k_candidates=kc, k=k, q_scale=qst, d_scale=dst,
                                  max_doc_len=w.ld_hi, workspace=ws)
    _, per = _time_loop(rerank, steps, 3, stream)
    ms = statistics.median(per)
    # what the scan competes with: exact FP16 scoring of every document, and
    # its stage 1 alone (the INT8 scan of every document, value only)
    s16 = torch.empty((w.n_q, w.n_docs), dtype=torch.float32, device=dev)
    _, per16 = _time_loop(lambda: m.maxsim_forward(Q16, ql, D16, cu, with_argmax=False, scores=s16), steps, 3, stream)
    _, per8 = _time_loop(lambda: m.maxsim_forward(Q8, ql, D8, cu, with_argmax=False, scores=s16, q_scale=qst,
                                                  d_scale=dst), steps, 3, stream)
    out["rerank_two_stage"] = {"n_q": w.n_q, "lq": w.lq, "n_docs": w.n_docs, "k_candidates": kc, "k": k,
                               "stage1": "int8 per tensor", "stage2": "fp16, corpus in HBM",
                               "call_ms": round(ms, 4), "queries_per_s": w.n_q / (ms / 1e3),
                               "fp16_exact_all_docs_value_only_ms": round(statistics.median(per16), 4),
                               "int8_scan_all_docs_value_only_ms": round(statistics.median(per8), 4)}
    del s16
    if m.maxsim_device_status() != 0:
        out["device_status"] = "fault"
    del Q8, D8, Q16, D16, ws
    torch.cuda.empty_cache()
    return out


CHAMFER_LANE_OPS_PER_PAIR = 7   # 3 sub, 1 mul, 2 fma, 1 min on the FP32 lanes


def _chamfer(m, sm_max_mhz, n=100_000, steps=10):
    """§4.2 "Generalization to Chamfer Distance" at the pages' 100K-point
    scale: one pair of 100,000-point clouds (uniform in the unit cube),
    forward (nearest neighbours both ways) and backward.  The search is
    bound by FP32 lane throughput: the roofline counts 7 lane operations per
    point pair against 128 FP32 lanes per SM at the maximum SM clock."""
    import torch
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    g = torch.Generator("cuda").manual_seed(0)
    P = torch.rand((n, 3), generator=g, device=dev)
    Q = torch.rand((n, 3), generator=g, device=dev)
    cu = torch.tensor([0, n], dtype=torch.int32, device=dev)
    fw = m.maxsim_chamfer_forward(P, cu, Q, cu)
    _, per = _time_loop(lambda: m.maxsim_chamfer_forward(P, cu, Q, cu, max_p=n, max_q=n), steps, 3, stream)
    ms = statistics.median(per)
    gcd = torch.ones(1, device=dev)
    _, perb = _time_loop(lambda: m.maxsim_chamfer_backward(gcd, P, cu, Q, cu, fw[2], fw[4]), steps, 3, stream)
    msb = statistics.median(perb)
    pairs = 2.0 * n * n
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    peak = sms * 128 * sm_max_mhz * 1e6 * 1e-12
    achieved = pairs * CHAMFER_LANE_OPS_PER_PAIR / (ms / 1e3) * 1e-12
    rec = {"points": [n, n], "fwd_ms": round(ms, 4), "bwd_ms": round(msb, 4), "pairs_per_s": pairs / (ms / 1e3),
           "roofline": {"bound": "alu", "achieved": round(achieved, 2), "peak": round(peak, 2),
                        "unit": "T FP32 lane-ops/s", "frac": round(achieved / peak, 3),
                        "peak_source": f"{sms} SMs x 128 FP32 lanes x {sm_max_mhz:.0f} MHz"}}
    if m.maxsim_device_status() != 0:
        rec["device_status"] = "fault"
    del P, Q
    torch.cuda.empty_cache()
    return rec


def _cpu_baseline(x, budget_s=15.0, threads=None):
    """The oracle, as it stands, on a bounded sample: the 16 queries against a
    prefix of the documents, on all host cores (one oracle call per chunk of
    pairs on a thread pool; the C code releases the GIL)."""
    import numpy as np

    import oracle
    from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
    threads = threads or (os.cpu_count() or 1)
    Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
    cu_h = cu.cpu().numpy()
    qb = syn.bits_u16(Q)
    ql_h = ql.cpu().numpy()

    def run(n_docs):
        Db = syn.bits_u16(D[: int(cu_h[n_docs])])
        t = time.perf_counter()
        oracle.forward_bits("fp16", qb, ql_h, Db, cu_h[: n_docs + 1], threads=threads)
        return time.perf_counter() - t

    n = 8
    dt = run(n)
    while dt < 1.0 and n < 4096:
        n *= 4
        dt = run(n)
    n = max(8, min(int(n * budget_s / max(dt, 1e-3)), 20000))
    dt = run(n)
    return {"value": n / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"16 queries x the first {n} of the 50,000 documents ({int(cu_h[n])} tokens), "
                      f"{dt:.1f} s"}


def run_ours(args):
    import torch

    import late_interaction_retrieval_maxsim_gb300 as m
    from late_interaction_retrieval_maxsim_gb300 import roofline as rl
    from late_interaction_retrieval_maxsim_gb300 import synthetic as syn

    world, rank, local = _dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    m.load_library()
    peaks = _peaks()
    w = rank_workload(syn.WORKLOADS[WORKLOAD], rank)
    x = syn.make_inputs(w, device="cuda")
    Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
    total = D.shape[0]
    scores = torch.empty((w.n_q, w.n_docs), dtype=torch.float32, device="cuda")
    argmax = torch.empty((w.n_q, w.n_docs, w.lq), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        m.maxsim_forward(Q, ql, D, cu, scores=scores, argmax=argmax)

    step()
    torch.cuda.synchronize()
    if m.maxsim_device_status() != 0:
        raise RuntimeError("device status word set after the first forward")

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total_ms, per = _time_loop(step, args.steps, args.warmup, stream, nvtx="timed")
    total_ms = max_over_ranks(total_ms, torch.device("cuda", local))
    if m.maxsim_device_status() != 0:
        raise RuntimeError("device status word set during the timed region")

    ms_per_step = total_ms / args.steps
    value = w.n_docs * world / (ms_per_step / 1e3)
    flops = rl.forward_flops(int(ql.sum()), total)
    kern_ms = statistics.mean(per)
    achieved = flops / (kern_ms / 1e3) / 1e12
    roof = {"bound": "tensor", "kernel": "maxsim_fwd_kernel", "achieved": achieved,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "peak_source": f"{peaks['source']} bf16 burst (FP16 runs at the same dense rate)",
            "algorithmic_flops_per_launch": flops,
            "traffic": _traffic(WORKLOAD),
            "algorithmic_bytes_per_launch": rl.forward_hbm_bytes(w.n_q, w.lq, w.n_docs, total)}

    # end to end through the public API with host-resident inputs: the queries
    # are copied in, the corpus streams from pinned host memory in blocks of
    # documents (maxsim_forward_host: the copy of a block overlaps the forward
    # of the previous one) and the scores are copied back, every step
    Qh = Q.cpu().pin_memory()
    Dh = D.cpu().pin_memory()
    qlh = ql.cpu().pin_memory()
    cuh = cu.cpu().pin_memory()
    sh = torch.empty(scores.shape, dtype=torch.float32).pin_memory()
    Qd, qld = torch.empty_like(Q), torch.empty_like(ql)
    block_docs = 5000
    block_tokens = block_docs * w.ld_hi
    hws = torch.empty(m.maxsim_forward_host_workspace_size(w.n_q, w.lq, w.n_docs, block_docs, block_tokens,
                                                           "fp16"), dtype=torch.uint8, device="cuda")

    def e2e_step():
        Qd.copy_(Qh, non_blocking=True)
        qld.copy_(qlh, non_blocking=True)
        m.maxsim_forward_host(Qd, qld, Dh, cuh, block_docs=block_docs, block_tokens=block_tokens,
                              with_argmax=True, scores=scores, argmax=argmax, workspace=hws)
        sh.copy_(scores, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, _ = _time_loop(e2e_step, e2e_steps, 2, stream)
    if m.maxsim_device_status() != 0:
        raise RuntimeError("device status word set during the end-to-end steps")
    h2d = sum(t.numel() * t.element_size() for t in (Qh, Dh, qlh, cuh))
    d2h = sh.numel() * sh.element_size()
    e2e = {"value": w.n_docs / (e2e_ms / e2e_steps / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "path": f"maxsim_forward_host: queries copied in, the corpus streamed from pinned host memory "
                   f"in {block_docs}-document blocks overlapped with the forward, scores copied back"}
    del hws

    extra = {}
    cpu = None
    if rank == 0 and world == 1:
        if not args.no_extra:
            extra = _extra_workloads(m, syn, rl, peaks)
            extra["chamfer_100k"] = _chamfer(m, clk.summary().get("sm_max_mhz") or 2070.0)
        cpu = _cpu_baseline(x, budget_s=args.cpu_budget)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
            "data": "synthetic: seeded N(0,1) token embeddings, L2-normalised, stored FP16",
            "config": {"workload": WORKLOAD, "n_q": w.n_q, "lq": w.lq, "n_docs_per_gpu": w.n_docs,
                       "ld": f"U[{w.ld_lo},{w.ld_hi}]", "total_tokens_per_gpu": total, "dim": 128,
                       "argmax": True,
                       "l2": f"inputs larger than L2 ({D.numel() * 2 / 1e9:.2f} GB of documents vs "
                             f"{L2_BYTES / 2**20:.0f} MiB L2), no flush needed",
                       "parallelism": f"doc-sharded x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * _forward_launches(w.lq, False),
            "clocks": clk.summary(),
            "extra": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------ single cases

# ``--case NAME``: one library entry point on seeded synthetic inputs, called
# ``--reps`` times on cuda:0 (no timing, no JSON line) -- the command the
# committed ncu summaries under profiles/ profile.

def _case_forward(m, syn, torch, a):
    w = syn.WORKLOADS[a.workload]
    x = syn.make_inputs(w, device="cuda", n_docs=a.n_docs)
    kw = dict(q_scale=x["q_scale"], d_scale=x["d_scale"])
    s, am, _ = m.maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], with_argmax=not a.value_only, **kw)
    for _ in range(a.reps - 1):
        m.maxsim_forward(x["Q"], x["q_lens"], x["D"], x["cu_seqlens"], with_argmax=not a.value_only, scores=s,
                         argmax=am, **kw)


def _case_int8_token(m, syn, torch, a):
    w = syn.WORKLOADS["int8_varlen"]
    n_docs = a.n_docs or w.n_docs
    cu = syn.cu_seqlens_from_lengths(syn.doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed)[:n_docs]).cuda()
    Q8, qs = syn.unit_tokens_int8_per_token(w.n_q * w.lq, w.dim, w.seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8_per_token(int(cu[-1]), w.dim, w.seed + 2, "cuda")
    ql = torch.full((w.n_q,), w.lq, dtype=torch.int32, device="cuda")
    for _ in range(a.reps):
        m.maxsim_forward_int8_per_token(Q8.view(w.n_q, w.lq, w.dim), qs.view(w.n_q, w.lq), ql, D8, ds, cu,
                                        with_argmax=not a.value_only)


def _case_backward(m, syn, torch, a):
    w = syn.WORKLOADS[a.workload]
    x = syn.make_inputs(w, device="cuda", n_docs=a.n_docs)
    Q, ql, D, cu = x["Q"], x["q_lens"], x["D"], x["cu_seqlens"]
    s, am, _ = m.maxsim_forward(Q, ql, D, cu)
    g = torch.softmax(s / 0.05, dim=1).contiguous()
    for _ in range(a.reps):
        m.maxsim_backward(g, am, Q, ql, D, cu)


def _case_chamfer(m, syn, torch, a):
    g = torch.Generator("cuda").manual_seed(0)
    P = torch.rand((a.points, 3), generator=g, device="cuda")
    Q = torch.rand((a.points, 3), generator=g, device="cuda")
    cu = torch.tensor([0, a.points], dtype=torch.int32, device="cuda")
    for _ in range(a.reps):
        _, _, apq, _, aqp = m.maxsim_chamfer_forward(P, cu, Q, cu)
        m.maxsim_chamfer_backward(torch.ones(1, device="cuda"), P, cu, Q, cu, apq, aqp)


def _case_rerank(m, syn, torch, a):
    """Two-stage scan on the INT8 varlen workload: 1,000 candidates, 100 kept."""
    w = syn.WORKLOADS["int8_varlen"]
    n_docs = a.n_docs or w.n_docs
    cu = syn.cu_seqlens_from_lengths(syn.doc_lengths(w.n_docs, w.ld_lo, w.ld_hi, w.seed)[:n_docs]).cuda()
    total = int(cu[-1])
    Q8, qs = syn.unit_tokens_int8(w.n_q * w.lq, w.dim, w.seed + 1, "cuda")
    D8, ds = syn.unit_tokens_int8(total, w.dim, w.seed + 2, "cuda")
    Q16 = syn.unit_tokens(w.n_q * w.lq, w.dim, w.seed + 1, "fp16", "cuda").view(w.n_q, w.lq, w.dim)
    D16 = syn.unit_tokens(total, w.dim, w.seed + 2, "fp16", "cuda")
    ql = torch.full((w.n_q,), w.lq, dtype=torch.int32, device="cuda")
    for _ in range(a.reps):
        m.maxsim_rerank_two_stage(Q8.view(w.n_q, w.lq, w.dim), D8, Q16, D16, ql, cu, k_candidates=1000, k=100,
                                  q_scale=qs, d_scale=ds, max_doc_len=w.ld_hi)


def _case_host(m, syn, torch, a):
    """Out-of-core forward: the ColBERT workload's corpus in pinned host
    memory, streamed in blocks of 5,000 documents."""
    w = syn.WORKLOADS["colbert_varlen"]
    x = syn.make_inputs(w, device="cuda", n_docs=a.n_docs)
    D_h = x["D"].cpu().pin_memory()
    cu_h = x["cu_seqlens"].cpu().pin_memory()
    for _ in range(a.reps):
        m.maxsim_forward_host(x["Q"], x["q_lens"], D_h, cu_h, block_docs=5000, block_tokens=5000 * w.ld_hi,
                              with_argmax=True)
    torch.cuda.synchronize()


CASES = {"forward": _case_forward, "int8-token": _case_int8_token, "backward": _case_backward,
         "chamfer": _case_chamfer, "rerank": _case_rerank, "host": _case_host}


def run_case(args) -> int:
    import torch

    import late_interaction_retrieval_maxsim_gb300 as m
    from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
    torch.cuda.set_device(0)
    m.load_library()
    CASES[args.case](m, syn, torch, args)
    torch.cuda.synchronize()
    status = m.maxsim_device_status()
    if status != 0:
        print(f"device status word {status:#x}", file=sys.stderr)
        return 1
    return 0


# ---------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle on the same workload: each step scores the 16 queries
    against a bounded block of documents (cycling through the corpus)."""
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from late_interaction_retrieval_maxsim_gb300 import synthetic as syn
    w = syn.WORKLOADS[WORKLOAD]
    threads = os.cpu_count() or 1
    block = args.ref_docs
    n_blocks = 8
    x = syn.make_inputs(w, device="cpu", n_docs=block * n_blocks)
    qb = syn.bits_u16(x["Q"])
    ql = x["q_lens"].numpy()
    cu = x["cu_seqlens"].numpy()
    Db = syn.bits_u16(x["D"])
    blocks = []
    for k in range(n_blocks):
        lo, hi = int(cu[k * block]), int(cu[(k + 1) * block])
        blocks.append((Db[lo:hi], (cu[k * block:(k + 1) * block + 1] - lo).astype(np.int32)))

    def step(k):
        d, c = blocks[k % n_blocks]
        oracle.forward_bits("fp16", qb, ql, d, c, threads=threads)

    for k in range(args.warmup):
        step(k)
    t = time.perf_counter()
    for k in range(args.steps):
        step(k)
    dt = time.perf_counter() - t
    ms = dt / args.steps * 1e3
    value = block / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded N(0,1) token embeddings, L2-normalised, stored FP16",
            "config": {"workload": WORKLOAD, "n_q": w.n_q, "lq": w.lq, "docs_per_step": block,
                       "ld": f"U[{w.ld_lo},{w.ld_hi}]", "dim": 128},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{block} documents per step x 16 queries, cycling over "
                                       f"the first {block * n_blocks} documents"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "torch": torch.__version__}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--ref-docs", type=int, default=32, help="documents per reference step")
    ap.add_argument("--case", choices=sorted(CASES), default=None,
                    help="run one entry point on synthetic inputs (for profilers) instead of the benchmark")
    ap.add_argument("--workload", default="colbert_varlen", help="--case: workload name (synthetic.WORKLOADS)")
    ap.add_argument("--n-docs", type=int, default=None, help="--case: first n documents of the workload")
    ap.add_argument("--points", type=int, default=20_000, help="--case chamfer: points per cloud")
    ap.add_argument("--reps", type=int, default=2, help="--case: calls of the entry point")
    ap.add_argument("--value-only", action="store_true", help="--case: forward without the argmax output")
    args = ap.parse_args()
    if args.case is not None:
        sys.exit(run_case(args))
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
