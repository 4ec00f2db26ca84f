"""Benchmark of the CSA2 hot path on GB300: one JSON line on rank 0.

Default workload: FP4-cache long-context decode (8 sequences x 2^20 entries, m=1,
MXFP4 indexer keys, FP4 main KV, 64 indexer heads, 64 core heads, top-512,
2048-block pool, 128-token window).  A step is one pass of the whole path for the
batch: write the new token's main-KV and indexer-K rows (compressor with m=1 +
FP4 / MXFP4 pack), full indexer scan with fused block max, block pool, candidate
rescoring, top-512, sparse shared-KV attention.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload fp4_decode_1M|decode_full_bf16|reindex_reuse_bf16]

With torchrun (N > 1) every rank runs the same per-GPU workload on its own
sequences (weak scaling, no data-path collective); time = max over ranks.
`--impl reference` times the CPU oracle (the only other implementation of the
path) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "decode queries/s & indexer entries/s at 1M ctx; % of HBM roofline (1 GB300)"
UNIT = "queries/s"


# ----------------------------------------------------------------------------- utils
def _env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _kernel_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "compressed_sparse_attention_06_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profile_traffic(name, src_hash):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source (matching hash); else None."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256_16") != src_hash:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    Q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        try:
            props = torch.cuda.get_device_properties(device)
            self.bus = getattr(props, "pci_bus_id", None)
        except Exception:
            self.bus = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        buses = sorted(set(r[0].strip() for r in rows))
        if self.bus is not None:
            sel = [r for r in rows if r[0].strip().lower().endswith(f"{self.bus:02x}:00.0")]
            rows = sel or rows
        if len(buses) > 1 and self.bus is None:
            rows = [r for r in rows if r[0].strip() == buses[0]]
        if not rows:
            return None
        sm = sorted(float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit())
        mx = max((float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- workloads
class FP4Decode:
    """FP4-cache long-context decode, B sequences x N entries."""
    name = "fp4_decode_1M"
    kernel_files = ("index_score_tc.cu", "index_score.cu", "sm100_ptx.cuh", "csa2_internal.cuh")
    profile = "index_score_fp4_decode_1M.txt"

    def __init__(self, B=8, N=1 << 20, seq0=0):
        self.B, self.N, self.seq0 = B, N, seq0
        self.H_I, self.H, self.k, self.window, self.block, self.n_keep = 64, 64, 512, 128, 8, 2048
        self.t = N - 1                        # query position; m = 1 so V = t entries are visible
        self.V = self.t

    def config(self):
        return {"workload": self.name, "batch": self.B, "context": self.N, "m": 1, "indexer_heads": self.H_I,
                "indexer_dim": 128, "heads": self.H, "head_dim": 512, "topk": self.k, "window": self.window,
                "pool": f"{self.n_keep} blocks of {self.block}",
                "cache": "main KV FP4 E2M1+E4M3/16 (288 B/entry), indexer K MXFP4 (68 B/entry)",
                "l2": "inputs larger than L2 (3.0 GB of caches per step)"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import csa2 as C
        from compressed_sparse_attention_06_gb300 import pipeline as P
        from compressed_sparse_attention_06_gb300 import workloads as W
        B, N = self.B, self.N
        self.kv = torch.empty((B, N, 288), dtype=torch.uint8, device=dev)
        self.ki = torch.empty((B, N, 68), dtype=torch.uint8, device=dev)
        chunk = 1 << 16
        for b in range(B):
            for r0 in range(0, N, chunk):
                n = min(chunk, N - r0)
                C.csa2_fp4_pack(W.fp4_rows("kv", self.seq0 + b, r0, n, N, dev), C.FP4_E4M3x16,
                                out=self.kv[b, r0:r0 + n])
                C.csa2_fp4_pack(W.fp4_rows("KI", self.seq0 + b, r0, n, N, dev), C.MXFP4_E8M0x32,
                                out=self.ki[b, r0:r0 + n])
        wl = W.fp4_decode(dev, B=B, N=N) if self.seq0 == 0 else _offset_workload(W.fp4_decode, dev, B, N,
                                                                                self.seq0)
        self.wl = wl
        self.qI, self.w, self.q, self.swa, self.sink = wl["qI"], wl["w"], wl["q"], wl["swa"], wl["sink"]
        self.C_new, self.Z_new, self.KI_new = wl["C_new"], wl["Z_new"], wl["KI_new"].reshape(B, 128)
        self.q_pos = wl.q_pos.clone()
        self.nv = P.visible_entries(self.q_pos, 1)
        self.pos_new = self.q_pos[:, 0].clone()
        self.buf = P.alloc_decode(B, 1, N, self.H, 512, dev, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()

    # the pieces of a step (all on the current stream)
    def write_new_rows(self):
        from compressed_sparse_attention_06_gb300 import csa2 as C
        t = self.t
        C.csa2_compress(self.C_new, self.Z_new, 1, pos0=self.pos_new, flags=C.W_ROPE,
                        out=self.kv[:, t], out_seq_stride=self.N)
        C.csa2_fp4_pack(self.KI_new, C.MXFP4_E8M0x32, out=self.ki[:, t], out_ld=self.N * 68)

    def scan(self):
        from compressed_sparse_attention_06_gb300 import csa2 as C
        C.csa2_index_score(self.qI, self.w, self.ki, self.nv, block=self.block, want_scores=False,
                           want_block_max=True, block_max=self.buf.block_max)

    def select_and_attend(self):
        from compressed_sparse_attention_06_gb300 import csa2 as C
        b = self.buf
        C.csa2_block_pool(b.block_max, self.nv, block=self.block, n_keep=self.n_keep, out=b.pool, ws=b.pool_ws)
        C.csa2_index_score(self.qI, self.w, self.ki, self.nv, pool=b.pool, block=self.block, scores=b.cand_scores)
        C.csa2_topk(b.cand_scores, self.nv, self.k, pool=b.pool, block=self.block, out_idx=b.idx, ws=b.topk_ws)
        C.csa2_sparse_attn(self.q, self.kv, b.idx, self.swa, self.q_pos, self.sink, window=self.window,
                           out=b.out, ws=b.attn_ws)

    launches_per_step = 10     # write x2, scan, pool x2, candidate scan, top-k x2, attention split + combine

    def scan_bytes(self):
        """Algorithmic bytes of one full-scan launch: every visible MXFP4 indexer row
        once, plus the queries and head weights."""
        return self.B * self.V * 68 + self.B * self.H_I * (128 * 2 + 4)

    def queries(self):
        return self.B

    def entries(self):
        return self.B * self.V

    # --- end to end through the public API with host buffers
    def e2e_inputs(self):
        pin = lambda t: t.detach().cpu().pin_memory()
        self.h_in = {"qI": pin(self.qI), "w": pin(self.w), "q": pin(self.q), "C_new": pin(self.C_new),
                     "Z_new": pin(self.Z_new), "KI_new": pin(self.KI_new),
                     "swa_row": pin(self.swa[:, self.t % 128].contiguous())}
        self.h_out = torch.empty(self.buf.out.shape, dtype=self.buf.out.dtype).pin_memory()
        self.h_idx = torch.empty(self.buf.idx.shape, dtype=self.buf.idx.dtype).pin_memory()
        self.d_swa_row = torch.empty_like(self.h_in["swa_row"], device=self.qI.device)
        return sum(v.numel() * v.element_size() for v in self.h_in.values()), \
            self.h_out.numel() * self.h_out.element_size() + self.h_idx.numel() * self.h_idx.element_size()

    def e2e_copy_in(self):
        self.qI.copy_(self.h_in["qI"], non_blocking=True)
        self.w.copy_(self.h_in["w"], non_blocking=True)
        self.q.copy_(self.h_in["q"], non_blocking=True)
        self.C_new.copy_(self.h_in["C_new"], non_blocking=True)
        self.Z_new.copy_(self.h_in["Z_new"], non_blocking=True)
        self.KI_new.copy_(self.h_in["KI_new"], non_blocking=True)
        self.swa[:, self.t % 128].copy_(self.h_in["swa_row"], non_blocking=True)

    def e2e_copy_out(self):
        self.h_out.copy_(self.buf.out, non_blocking=True)
        self.h_idx.copy_(self.buf.idx, non_blocking=True)

    # --- the oracle on a bounded sample (host cores)
    def oracle_prepare(self, b=0):
        """Host copies of one sequence's packed caches (taken outside any timing)."""
        from compressed_sparse_attention_06_gb300 import workloads as W
        from oracle import csa2_oracle as O
        N = self.N
        ki = torch.cat([W.fp4_rows("KI", self.seq0 + b, r0, min(1 << 18, N - r0), N, "cpu")
                        for r0 in range(0, N, 1 << 18)]).numpy()
        self.o_ki = O.mxfp4_pack(ki)
        wl = self.wl if hasattr(self, "wl") else None
        if wl is None:
            wl = W.fp4_decode("cpu", B=self.B, N=N)
        self.o_q = dict(qI=wl["qI"][b, 0].double().cpu().numpy(), w=wl["w"][b, 0].double().cpu().numpy(),
                        q=wl["q"][b, 0].double().cpu().numpy(), swa=wl["swa"][b].double().cpu().numpy(),
                        sink=wl["sink"].double().cpu().numpy())
        self.o_b = b
        # the main-KV rows the query selects, packed, so the timed part only gathers them
        V = self.V
        sc = O.index_score(self.o_q["qI"], self.o_q["w"], O.mxfp4_unpack(self.o_ki[:V]), V)
        idx = O.topk(sc, V, self.k)
        self.o_kv = {int(s): O.nvfp4_pack(W.fp4_rows("kv", self.seq0 + b, int(s), 1, N, "cpu").numpy())
                     for s in idx if s >= 0}

    def oracle_query(self):
        """One query of the step through the oracle: dequantise the indexer cache, score,
        block max, pool, top-512 inside the pool, gather + dequantise the selected
        main-KV rows, attend."""
        from oracle import csa2_oracle as O
        o = self.o_q
        V = self.V
        K = O.mxfp4_unpack(self.o_ki[:V])
        sc = O.index_score(o["qI"], o["w"], K, V)
        pool = O.block_pool(O.block_max(sc, V, self.block), V, self.block, self.n_keep)
        idx = O.reindex_topk(sc, pool, V, self.k)
        kv_sel = _RowMap({int(s): O.nvfp4_unpack(self.o_kv[int(s)])[0] for s in idx if s >= 0})
        out, lse, _ = O.sparse_attn(o["q"], kv_sel, idx, o["swa"], 0, self.t, o["sink"], self.window)
        return out


class _RowMap:
    """Indexable view over a dict of gathered rows (the oracle indexes kv[s])."""

    def __init__(self, rows):
        self.rows = rows
        self.shape = (max(rows) + 1 if rows else 0, 512)

    def __getitem__(self, s):
        return self.rows[int(s)]


def _offset_workload(fn, dev, B, N, seq0):
    """The workload for sequences seq0 .. seq0+B-1: draw seq0+B sequences' query-side
    tensors and keep the last B (ranks > 0 under torchrun)."""
    wl = fn(dev, B=seq0 + B, N=N)
    for k, v in list(wl.tensors.items()):
        if v.dim() and v.shape[0] == seq0 + B:
            wl.tensors[k] = v[seq0:].contiguous()
    wl.q_pos = wl.q_pos[seq0:].contiguous()
    wl.B = B
    return wl


WORKLOADS = {"fp4_decode_1M": FP4Decode}


def _make(args, seq0=0):
    kw = {"seq0": seq0}
    if args.n_ctx:
        kw["N"] = args.n_ctx
    return WORKLOADS[args.workload](**kw)


# ----------------------------------------------------------------------------- arms
def run_ours(args):
    rank, world, local = _env_rank()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from compressed_sparse_attention_06_gb300 import build_lib
    if rank == 0 or world == 1:
        build_lib.build()
    if dist is not None:
        dist.barrier()
    from compressed_sparse_attention_06_gb300 import csa2 as C
    C.load()
    wl = _make(args, seq0=rank * 8)
    wl.setup(dev)
    stream = torch.cuda.current_stream(dev)

    # warm-up (also sets kernel attributes before any graph capture)
    for _ in range(max(1, args.warmup)):
        wl.write_new_rows()
        wl.scan()
        wl.select_and_attend()
    C.csa2_ctx_check()
    g_pre = g_post = None
    if not args.no_graph:
        g_pre, g_post = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g_pre, stream=s):
                wl.write_new_rows()
            with torch.cuda.graph(g_post, stream=s):
                wl.select_and_attend()
        stream.wait_stream(s)
        for _ in range(2):
            g_pre.replay(); wl.scan(); g_post.replay()
    torch.cuda.synchronize()

    def step(ev0=None, ev1=None):
        if g_pre is not None:
            g_pre.replay()
        else:
            wl.write_new_rows()
        if ev0 is not None:
            ev0.record(stream)
        wl.scan()
        if ev1 is not None:
            ev1.record(stream)
        if g_post is not None:
            g_post.replay()
        else:
            wl.select_and_attend()

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0.record(stream)
    for i in range(K):
        step(*evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    C.csa2_ctx_check()
    ms_total = t0.elapsed_time(t1)
    scan_ms = sum(a.elapsed_time(b) for a, b in evs) / K
    if dist is not None:
        tt = torch.tensor([ms_total, scan_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_total, scan_ms = float(tt[0]), float(tt[1])
    ms_step = ms_total / K

    # end to end: host inputs -> device, step, result -> host, every step
    h2d, d2h = wl.e2e_inputs()
    torch.cuda.synchronize()
    for _ in range(2):
        wl.e2e_copy_in(); step(); wl.e2e_copy_out(); torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = time.perf_counter()
    for _ in range(K):
        wl.e2e_copy_in()
        step()
        wl.e2e_copy_out()
        torch.cuda.synchronize()
    e_s = time.perf_counter() - e0
    if dist is not None:
        tt = torch.tensor([e_s], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e_s = float(tt[0])

    hbm, bf16, bf16s, src = _peaks()
    achieved = wl.scan_bytes() / (scan_ms * 1e-3) / 1e9
    traffic = _profile_traffic(wl.profile, _kernel_hash(wl.kernel_files))
    value = world * wl.queries() / (ms_step * 1e-3)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32", "data": "synthetic (seeded counter-based generator)",
        "config": {**wl.config(), "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "cuda_graph": g_pre is not None},
        "entries_per_s": world * wl.entries() / (ms_step * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "kernel": "csa2_index_score (full scan, fused block max)",
                     "kernel_ms": scan_ms, "bytes_per_launch": wl.scan_bytes(), "peak_source": src},
        "e2e": {"value": world * wl.queries() * K / e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": wl.launches_per_step * K,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, args)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def cpu_baseline(wl, args, n_queries=None):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    import numpy as np
    wl.oracle_prepare(0)
    n = n_queries or args.cpu_queries
    t0 = time.perf_counter()
    for _ in range(n):
        wl.oracle_query()
    dt = time.perf_counter() - t0
    try:
        import threadpoolctl
        cores = max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()) or 1
    except Exception:
        cores = os.cpu_count() or 1
    return {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} query(ies) of sequence 0 (full pipeline per query: MXFP4 dequant of all "
                      f"{wl.V} indexer rows, f64 scores, block max, pool, top-512, FP4 row gather, attention); "
                      f"numpy f64, BLAS threads for the score matmul, {os.uname().machine}"}


def run_reference(args):
    rank, world, _ = _env_rank()
    if rank != 0:
        return
    wl = _make(args)
    wl.oracle_prepare(0)
    for _ in range(args.warmup):
        wl.oracle_query()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        wl.oracle_query()
    dt = time.perf_counter() - t0
    v = args.steps / dt
    try:
        import threadpoolctl
        cores = max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()) or 1
    except Exception:
        cores = os.cpu_count() or 1
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
           "config": wl.config(),
           "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": "each step = one query of sequence 0 through the whole oracle pipeline"},
           "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="fp4_decode_1M", choices=sorted(WORKLOADS))
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-queries", type=int, default=3)
    ap.add_argument("--n-ctx", type=int, default=None, help="override the context length (quick checks only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
