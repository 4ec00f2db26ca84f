"""Benchmark of the CSA2 hot path on GB300: one JSON line on rank 0.

Default workload: FP4-cache long-context decode (8 sequences x 2^20 entries, m=1,
MXFP4 indexer keys, FP4 main KV, 64 indexer heads, 64 core heads, top-512,
2048-block pool, 128-token window).  A step is one pass of the whole path for the
batch: write the new token's main-KV and indexer-K rows (compressor with m=1 +
FP4 / MXFP4 pack), full indexer scan with fused block max, block pool, candidate
rescoring, top-512, sparse shared-KV attention.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload fp4_decode_1M|decode_full_bf16|reindex_reuse_bf16|
                              prefill_chunk_bf16|tiny_full_layer_fp32|hca_decode_1M|compress_step_m4|
                              fp4_decode_1M_v4pro|prefill_varlen_compress]

Besides the step rate, the line carries each stage's time (timed separately with
CUDA events after the main loop) against its own roofline.  With torchrun (N > 1)
every rank runs the same per-GPU workload on its own sequences (weak scaling, no
data-path collective); time = max over ranks.  `--impl reference` times the CPU
oracle (the only other implementation of the path) on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "decode queries/s & indexer entries/s at 1M ctx; % of HBM roofline (1 GB300)"
UNIT = "queries/s"
FP4_PER_BF16 = 13.5 / 2.25      # nominal dense tensor rates per GPU, FP4 over bf16


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


def _cores():
    try:
        import threadpoolctl
        return max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()) or 1
    except Exception:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    Q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        try:
            self.bus = getattr(torch.cuda.get_device_properties(device), "pci_bus_id", None)
        except Exception:
            self.bus = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
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
                "samples": len(rows), "window": "warm-up and timed steps"}


def _C():
    from compressed_sparse_attention_06_gb300 import csa2
    return csa2


# ----------------------------------------------------------------------------- workloads
class Workload:
    """A step = pre() ; main() ; post().  main() is the kernel the roofline entry
    describes (timed with CUDA events inside every timed step); pre/post are
    captured in CUDA graphs.  stages() lists (name, fn, bytes, flops) for the
    separate per-stage timing."""
    name = ""
    main_name = ""
    main_bound = "hbm"
    kernel_files = ("index_score_tc.cu", "index_score.cu", "sm100_ptx.cuh", "csa2_internal.cuh")
    profile = None
    flush_l2 = False          # True: the step's data fit in L2, flush it before every timed step
    dtype = "f16/bf16 MMA, fp32 accumulate"

    def pre(self):
        pass

    def side(self):
        """Work of the step that nothing later in the step reads (cache rows written for
        the next steps): it runs on a second stream once the scan is done, beside the
        selections and the attention, and the step ends only when it has finished."""
        pass

    has_side = False

    def post(self):
        pass

    def stages(self):
        return []

    def launches_per_step(self):
        return 0

    # generic end-to-end: refresh e2e_in from pinned host copies, read e2e_out back
    def e2e_inputs(self):
        self.h_in = [(t, t.detach().cpu().pin_memory()) for t in self.e2e_in]
        self.h_out = [(t, torch.empty(t.shape, dtype=t.dtype).pin_memory()) for t in self.e2e_out]
        return (sum(h.numel() * h.element_size() for _, h in self.h_in),
                sum(h.numel() * h.element_size() for _, h in self.h_out))

    def e2e_copy_in(self):
        for d, h in self.h_in:
            d.copy_(h, non_blocking=True)

    def e2e_copy_out(self):
        for d, h in self.h_out:
            h.copy_(d, non_blocking=True)


class FP4Decode(Workload):
    """FP4-cache long-context decode, B sequences x N entries (the headline)."""
    name = "fp4_decode_1M"
    main_name = "csa2_index_score (FP4 QK full scan over MXFP4 keys, fused block max)"
    profile = "index_score_fp4_decode_1M.txt"
    kernel_files = ("index_scan_fp4.cu", "index_score.cu", "index_score_tc.cuh", "sm100_ptx.cuh", "csa2_internal.cuh")
    dtype = ("indexer QK MXFP4 x MXFP4 (tcgen05 kind::mxf4, E8M0 block scales, fp32 accumulate); "
             "attention bf16 MMA over FP4 E2M1+E4M3 rows, fp32 accumulate")

    H, K = 64, 512                            # query heads, top-k

    def __init__(self, B=8, N=1 << 20, seq0=0):
        self.B, self.N, self.seq0 = B, N, seq0
        self.H_I, self.window, self.block, self.n_keep = 64, 128, 8, 2048
        self.k = self.K
        self.n_top = (self.k + 31) // 32 * 32     # blocks rescored for the top-k
        self.t = N - 1                        # query position; m = 1 so V = t entries are visible
        self.V = self.t

    def config(self):
        return {"workload": self.name, "batch": self.B, "context": self.N, "m": 1, "indexer_heads": self.H_I,
                "indexer_dim": 128, "heads": self.H, "head_dim": 512, "topk": self.k, "window": self.window,
                "pool": f"{self.n_keep} blocks of {self.block}",
                "cache": "main KV FP4 E2M1+E4M3/16 (288 B/entry), indexer K MXFP4 (68 B/entry)",
                "l2": f"inputs larger than L2 ({self.B * self.N * 356 / 1e9:.1f} GB of caches per step)"}

    def setup(self, dev):
        C = _C()
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
        wl = W.fp4_decode(dev, B=B, N=N, H=self.H) if self.seq0 == 0 else \
            _offset_workload(lambda d, B, N: W.fp4_decode(d, B=B, N=N, H=self.H), dev, B, N, self.seq0)
        self.wl = wl
        self.qI, self.w, self.q, self.swa, self.sink = wl["qI"], wl["w"], wl["q"], wl["swa"], wl["sink"]
        self.C_new, self.Z_new, self.KI_new = wl["C_new"], wl["Z_new"], wl["KI_new"].reshape(B, 128)
        self.q_pos = wl.q_pos.clone()
        self.nv = P.visible_entries(self.q_pos, 1)
        self.pos_new = self.q_pos[:, 0].clone()
        self.buf = P.alloc_decode(B, 1, N, self.H, 512, dev, out_dtype=torch.bfloat16, k=self.k)
        self.qI_mx = self.buf.qI_mx
        self.swa_row = self.swa[:, self.t % 128]
        self.e2e_in = [self.qI, self.w, self.q, self.C_new, self.Z_new, self.KI_new]
        self.e2e_out = [self.buf.out, self.buf.idx]
        torch.cuda.synchronize()

    def e2e_inputs(self):
        # the step's inputs become views of one device buffer (256-byte aligned), so one
        # copy from one pinned host buffer refreshes them all; the window row lives in
        # the ring and is copied on its own
        names = ["qI", "w", "q", "C_new", "Z_new", "KI_new"]
        ts = [getattr(self, n) for n in names]
        offs, tot = [], 0
        for t in ts:
            offs.append(tot)
            tot += (t.numel() * t.element_size() + 255) // 256 * 256
        self.in_buf = torch.empty(tot, dtype=torch.uint8, device=ts[0].device)
        for n, t, o in zip(names, ts, offs):
            v = self.in_buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            v.copy_(t)
            setattr(self, n, v)
        self.e2e_in = [self.in_buf]
        # the step's results (attention output, selected indices) likewise share one
        # buffer, read back with one copy
        b = self.buf
        ob = b.out.numel() * b.out.element_size()
        ob_pad = (ob + 255) // 256 * 256
        self.out_buf = torch.empty(ob_pad + b.idx.numel() * b.idx.element_size(), dtype=torch.uint8,
                                   device=b.out.device)
        b.out = self.out_buf[:ob].view(b.out.dtype).view(b.out.shape)
        b.idx = self.out_buf[ob_pad:].view(b.idx.dtype).view(b.idx.shape)
        self.e2e_out = [self.out_buf]
        torch.cuda.synchronize()
        h2d, d2h = super().e2e_inputs()
        self.h_swa = self.swa_row.detach().cpu().pin_memory()
        return h2d + self.h_swa.numel() * self.h_swa.element_size(), d2h

    def e2e_copy_in(self):
        super().e2e_copy_in()
        self.swa_row.copy_(self.h_swa, non_blocking=True)      # the new token's window row

    # stages
    def write(self):
        self.write_rows()

    def write_rows(self):
        """The new token's main-KV and indexer-key rows (entry t; the step's query sees
        entries 0 .. t-1, so only later steps read them)."""
        C = _C()
        t = self.t
        C.csa2_compress(self.C_new, self.Z_new, 1, pos0=self.pos_new, flags=C.W_ROPE, out=self.kv[:, t],
                        out_seq_stride=self.N)
        C.csa2_fp4_pack(self.KI_new, C.MXFP4_E8M0x32, out=self.ki[:, t], out_ld=self.N * 68)


    def main(self):
        # the FP4 QK path with the bf16 query packed to MXFP4 inside the scan (the packed
        # bytes kept for the candidate scan of the top-1024 path); every score is stored
        # only for the fused selection, which reads those of the best blocks
        fused = self.fused_select()
        _C().csa2_index_score_mxq(self.qI, self.w, self.ki, self.nv, block=self.block,
                                  scores=self.buf.scores if fused else None, want_scores=fused,
                                  want_block_max=True, block_max=self.buf.block_max,
                                  block_hist=self.buf.block_hist, q_mx_out=self.qI_mx)

    def fused_select(self):
        from compressed_sparse_attention_06_gb300 import pipeline as P
        return P.pool_topk_applies(self.k, self.block, self.n_keep, self.buf.block_max.shape[-1])

    def select(self):
        """The pool and the layer's top-k: one cluster kernel from the stored scores of
        the k best blocks where that kernel takes the shape (k * block <= 4,096), else
        the pool with its best-block list, the candidate scan of those blocks and the
        cluster top-k (V4-Pro's top-1024)."""
        b = self.buf
        if self.fused_select():
            _C().csa2_pool_topk(b.block_max, b.block_hist, b.scores, self.nv, self.k, block=self.block,
                                n_keep=self.n_keep, out=b.pool, out_idx=b.idx)
        else:
            self.pool(); self.cand(); self.topk()

    def scan_bf16_query(self):
        """The other reading of the pages: the bf16 indexer query over the same MXFP4
        keys (keys dequantised exactly to f16 in tensor memory, f16 MMA).  Timed as a
        stage for comparison; the step runs the FP4 QK path."""
        if not hasattr(self, "bmax_bf16q"):
            self.bmax_bf16q = torch.empty_like(self.buf.block_max)
        _C().csa2_index_score(self.qI, self.w, self.ki, self.nv, block=self.block, want_scores=False,
                              want_block_max=True, block_max=self.bmax_bf16q)

    def pool(self):
        b = self.buf
        _C().csa2_block_pool(b.block_max, self.nv, block=self.block, n_keep=self.n_keep, out=b.pool, ws=b.pool_ws,
                             block_hist=b.block_hist, n_top=b.top_blocks.shape[-1], out_top=b.top_blocks)

    def cand(self):
        b = self.buf
        _C().csa2_index_score(self.qI_mx, self.w, self.ki, self.nv, pool=b.top_blocks, block=self.block,
                              scores=b.cand_scores)

    def topk(self):
        b = self.buf
        _C().csa2_topk(b.cand_scores, self.nv, self.k, pool=b.top_blocks, block=self.block, out_idx=b.idx,
                       ws=b.topk_ws)

    def attn(self, prepared=False):
        b = self.buf
        C = _C()
        _C().csa2_sparse_attn(self.q, self.kv, b.idx, self.swa, self.q_pos, self.sink, window=self.window, out=b.out,
                              ws=b.attn_ws, flags=C.ATTN_DEFAULT | (C.ATTN_PREPARED if prepared else 0))

    def prepare(self):
        """The attention's query half (depends only on q and its position)."""
        _C().csa2_attn_prepare(self.q, self.q_pos, self.buf.attn_ws, self.k, window=self.window, N=self.N,
                               swa_cap=128)

    def pre(self):
        pass

    has_side = True

    def side(self):
        self.write_rows()

    def post(self):
        self.select(); self.attn()

    def launches_per_step(self):
        # compress, the new indexer-key row's pack, histogram zeroing, scan (packing the
        # query), pool + top-k (or pool, candidate scan, top-k), then per 64-head pass of
        # the attention: query prep, attention (its key splits merged in the kernel)
        return (5 if self.fused_select() else 7) + 2 * ((self.H + 63) // 64)

    def main_amount(self):
        """Algorithmic bytes of one full-scan launch: every visible MXFP4 indexer row
        once, plus the bf16 queries and the head weights."""
        return self.B * self.V * 68 + self.B * self.H_I * (256 + 4)

    def stages(self):
        B, H = self.B, self.H
        attn_bytes = B * (self.k * 288 + self.window * 1024 + H * 512 * 2 * 2)
        attn_flops = B * H * (self.k + self.window) * 512 * 4
        extra = []
        if self.H <= 64:
            extra = [("sparse attention (query half prepared)", lambda: self.attn(prepared=True), attn_bytes, attn_flops),
                     ("attention query half", self.prepare, B * H * 512 * 2 * 2, 0)]
        return [("write new rows", self.write, B * (2 * 1024 + 256 + 288 + 68 + self.H_I * (256 + 68)), 0),
                ("index scan", self.main, self.main_amount(), 2 * B * self.V * 64 * 128, "fp4"),
                ("index scan (bf16 q)", self.scan_bf16_query, B * self.V * 68 + B * self.H_I * (256 + 4),
                 2 * B * self.V * 64 * 128, "bf16"),
                (f"pool + top-{self.k}", self.select, B * ((self.V + 7) // 8) * 4 + B * self.n_top * 8 * 4, 0),
                ("block pool alone", self.pool, B * ((self.V + 7) // 8) * 4, 0),
                ("sparse attention", self.attn, attn_bytes, attn_flops)] + extra

    def queries(self):
        return self.B

    def entries(self):
        return self.B * self.V

    # --- the oracle on a bounded sample (host cores)
    def oracle_prepare(self, b=0):
        """Host copies of one sequence's packed caches (taken outside any timing): the
        MXFP4 indexer rows, the packed indexer query, and the FP4 main-KV rows of the
        entries the query selects (the timed part dequantises only those)."""
        from compressed_sparse_attention_06_gb300 import workloads as W
        from oracle import csa2_oracle as O
        from oracle import native as NO
        N, V = self.N, self.V
        ki = torch.cat([W.fp4_rows("KI", self.seq0 + b, r0, min(1 << 18, N - r0), N, "cpu")
                        for r0 in range(0, N, 1 << 18)]).numpy()
        self.o_ki = NO.mxfp4_pack(ki)
        wl = self.wl if hasattr(self, "wl") else W.fp4_decode("cpu", B=self.B, N=N)
        self.o_qmx = NO.mxfp4_pack(wl["qI"][b, 0].float().cpu().numpy())
        self.o_q = dict(w=wl["w"][b, 0].double().cpu().numpy(), q=wl["q"][b, 0].double().cpu().numpy(),
                        swa=wl["swa"][b].double().cpu().numpy(), sink=wl["sink"].double().cpu().numpy())
        # the selection is the top-k of all scores (the pool lemma), so the rows to hand
        # over are known before the timed queries
        sc = O.index_score(NO.mxfp4_unpack(self.o_qmx), self.o_q["w"], NO.mxfp4_unpack(self.o_ki[:V]), V)
        ids = O.topk(sc, V, self.k)
        self.o_ids = ids[ids >= 0]
        self.o_kv = np.concatenate([NO.nvfp4_pack(W.fp4_rows("kv", self.seq0 + b, int(s), 1, N, "cpu").numpy())
                                    for s in self.o_ids])
        self.o_threads = os.cpu_count() or 1

    def oracle_query(self):
        """One query of the step through the C++ oracle: MXFP4 dequantisation and
        score of every visible indexer row (split over the host's cores), block max,
        pool, top-k inside the pool, FP4 dequantisation of the selected main-KV rows,
        attention with the window and the sink."""
        from oracle import native as NO
        o = self.o_q
        out, lse, idx = NO.decode_query_fp4(self.o_ki, self.V, self.o_qmx, o["w"], self.o_ids, self.o_kv, o["q"],
                                            o["swa"], 0, self.t, o["sink"], block=self.block, n_keep=self.n_keep,
                                            k=self.k, window=self.window, threads=self.o_threads)
        return out

    def oracle_cores(self):
        return self.o_threads

    def oracle_sample_text(self, n):
        return (f"{n} query(ies) of sequence 0 through the C++ oracle (f64; per query: MXFP4 dequant + score of all "
                f"{self.V} indexer rows over {self.o_threads} std::threads, block max, pool, top-{self.k} inside "
                f"the pool, FP4 dequant of the selected rows, attention), {os.uname().machine}")


class V4ProDecode(FP4Decode):
    """The FP4 decode step with the V4-Pro configuration of the DSA-to-CSA/HCA page's
    table («两个已公开配置»): CSA top-1024 and 128 query heads (64 indexer heads)."""
    name = "fp4_decode_1M_v4pro"
    H, K = 128, 1024


class DecodeBF16(Workload):
    """Decoder Full-mode decode, bf16, batch 32 x 64K, with the pool."""
    name = "decode_full_bf16"
    main_name = "csa2_index_score (bf16 full scan, fused block max)"

    def __init__(self, B=32, N=65536, seq0=0):
        self.B, self.N = B, N
        self.H_I, self.H, self.k, self.window, self.block, self.n_keep = 64, 64, 512, 128, 8, 2048
        self.t, self.V = N - 1, N - 1

    def config(self):
        return {"workload": self.name, "batch": self.B, "context": self.N, "m": 1, "indexer_heads": self.H_I,
                "heads": self.H, "topk": self.k, "window": self.window, "pool": f"{self.n_keep} blocks of 8",
                "cache": "bf16 main KV and indexer K", "l2": "inputs larger than L2 (2.5 GB of caches)"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import pipeline as P
        from compressed_sparse_attention_06_gb300 import workloads as W
        wl = W.decode_full_bf16(dev, B=self.B, N=self.N)
        self.wl = wl
        self.kv, self.KI, self.qI, self.w, self.q = wl["kv"], wl["KI"], wl["qI"], wl["w"], wl["q"]
        self.swa, self.sink, self.C_new, self.Z_new = wl["swa"], wl["sink"], wl["C_new"], wl["Z_new"]
        self.q_pos = wl.q_pos.clone()
        self.pos_new = self.q_pos[:, 0].clone()
        self.nv = P.visible_entries(self.q_pos, 1)
        self.buf = P.alloc_decode(self.B, 1, self.N, self.H, 512, dev)
        self.e2e_in = [self.qI, self.w, self.q, self.C_new, self.Z_new]
        self.e2e_out = [self.buf.out, self.buf.idx]

    def write(self):
        C = _C()
        C.csa2_compress(self.C_new, self.Z_new, 1, pos0=self.pos_new, flags=C.W_ROPE, out=self.kv[:, self.t],
                        out_seq_stride=self.N)

    def main(self):
        _C().csa2_index_score(self.qI, self.w, self.KI, self.nv, scores=self.buf.scores, want_block_max=True,
                              block_max=self.buf.block_max, block_hist=self.buf.block_hist)

    def select(self):
        b = self.buf
        _C().csa2_pool_topk(b.block_max, b.block_hist, b.scores, self.nv, self.k, n_keep=self.n_keep, out=b.pool,
                            out_idx=b.idx)

    def pool(self):
        b = self.buf
        _C().csa2_block_pool(b.block_max, self.nv, n_keep=self.n_keep, out=b.pool, ws=b.pool_ws,
                             block_hist=b.block_hist, n_top=b.top_blocks.shape[-1], out_top=b.top_blocks)

    def cand(self):
        b = self.buf
        _C().csa2_index_score(self.qI, self.w, self.KI, self.nv, pool=b.top_blocks, scores=b.cand_scores)

    def topk(self):
        b = self.buf
        _C().csa2_topk(b.cand_scores, self.nv, self.k, pool=b.top_blocks, out_idx=b.idx, ws=b.topk_ws)

    def attn(self):
        b = self.buf
        _C().csa2_sparse_attn(self.q, self.kv, b.idx, self.swa, self.q_pos, self.sink, out=b.out, ws=b.attn_ws)

    def pre(self):
        self.write()

    def post(self):
        self.select(); self.attn()

    def launches_per_step(self):
        return 8          # compress, zeroing, scan, histogram, pool + top-k, query prep, attention, combine

    def main_amount(self):
        return self.B * self.V * 256 + self.B * self.H_I * (128 * 2 + 4)

    def stages(self):
        B, H = self.B, self.H
        return [("write new row", self.write, B * 3 * 1024, 0),
                ("index scan", self.main, self.main_amount(), 2 * B * self.V * 64 * 128),
                ("pool + top-512", self.select, B * (self.V // 8) * 4 + B * 4096 * 4, 0),
                ("sparse attention", self.attn, B * (640 * 1024 + H * 512 * 4), B * H * 640 * 512 * 4)]

    def queries(self):
        return self.B

    def entries(self):
        return self.B * self.V


class ReindexReuse(Workload):
    """Reindex over the pooled 16,384 candidates + 3 Reuse layers, bf16, 64 x 256K."""
    name = "reindex_reuse_bf16"
    main_name = "csa2_index_score (bf16 candidate scan, 16,384 pooled entries per query)"

    def __init__(self, B=64, N=262144, seq0=0):
        self.B, self.N = B, N
        self.t, self.V = N - 1, N - 1

    def config(self):
        return {"workload": self.name, "batch": self.B, "context": self.N, "m": 1, "indexer_heads": 64,
                "heads": 64, "topk": 512, "window": 128, "pool": "2048 given blocks of 8 (16,384 candidates)",
                "layers": "Reindex + 3 Reuse", "l2": "inputs larger than L2 (20 GB of caches)"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import pipeline as P
        from compressed_sparse_attention_06_gb300 import workloads as W
        C = _C()
        wl = W.reindex_reuse_bf16(dev, B=self.B, N=self.N)
        self.wl = wl
        self.nv = P.visible_entries(wl.q_pos, 1)
        self.q_pos = wl.q_pos
        self.cand_scores = torch.empty((self.B, 1, 16384), dtype=torch.float32, device=dev)
        self.idx = torch.empty((self.B, 1, 512), dtype=torch.int32, device=dev)
        self.outs = [torch.empty((self.B, 1, 64, 512), dtype=torch.bfloat16, device=dev) for _ in range(4)]
        self.topk_ws = C._ws(C.csa2_topk_workspace_bytes(self.B, 16384, 512), dev)
        self.attn_ws = C._ws(C.csa2_sparse_attn_workspace_bytes(self.B, 1, 64, 512, 128, N=self.N, swa_cap=128), dev)
        self.e2e_in = [wl["qI"], wl["w"]] + [wl[f"q{l}"] for l in range(4)]
        self.e2e_out = self.outs + [self.idx]

    def main(self):
        wl = self.wl
        _C().csa2_index_score(wl["qI"], wl["w"], wl["KI"], self.nv, pool=wl["pool"], scores=self.cand_scores)

    def topk(self):
        _C().csa2_topk(self.cand_scores, self.nv, 512, pool=self.wl["pool"], out_idx=self.idx, ws=self.topk_ws)

    def attn_layer(self, l):
        wl = self.wl
        _C().csa2_sparse_attn(wl[f"q{l}"], wl["kv"], self.idx, wl[f"swa{l}"], self.q_pos, wl["sink"],
                              out=self.outs[l], ws=self.attn_ws)

    def post(self):
        self.topk()
        for l in range(4):
            self.attn_layer(l)

    def launches_per_step(self):
        return 1 + 2 + 4 * 2

    def main_amount(self):
        return self.B * 16384 * 256 + self.B * 64 * (128 * 2 + 4)

    def stages(self):
        B = self.B
        st = [("candidate scan", self.main, self.main_amount(), 2 * B * 16384 * 64 * 128),
              ("top-512", self.topk, B * 16384 * 4, 0)]
        for l in range(4):
            st.append((f"attention layer {l}", (lambda l=l: self.attn_layer(l)), B * (640 * 1024 + 64 * 512 * 4),
                       B * 64 * 640 * 512 * 4))
        return st

    def queries(self):
        return self.B

    def entries(self):
        return self.B * 16384


class HCADecode(Workload):
    """HCA layer decode (DSA-to-CSA/HCA page, «HCA：公式 (20)–(26)»): 8 sequences at
    1M tokens, m' = 128 -> 8,192 FP4 compressed entries each; the step writes the
    entry completed by the new token (decode compressor with its state) and attends
    densely over every visible entry plus the 128-token window."""
    name = "hca_decode_1M"
    main_name = "csa2_dense_attn (tcgen05, 8,191 FP4 entries + 128 window rows per query)"
    main_bound = "tensor"
    kernel_files = ("attn_tc.cu", "attn.cu", "sm100_ptx.cuh", "csa2_internal.cuh")
    flush_l2 = True

    def __init__(self, B=8, N=1 << 20, seq0=0):
        self.B, self.tokens, self.seq0 = B, N, seq0
        self.m = 128
        self.N = N // self.m                  # HCA entries in the cache
        self.t = N - 1                        # the new token completes block N/m - 1
        self.V = self.t // self.m             # entries visible to the query (the new one is not)
        self.H = 64

    def config(self):
        return {"workload": self.name, "batch": self.B, "context_tokens": self.tokens, "m": self.m,
                "entries": self.N, "heads": self.H, "head_dim": 512, "window": 128, "attention": "dense over all "
                "visible entries (no indexer)", "cache": "main KV FP4 E2M1+E4M3/16 (288 B/entry)",
                "l2": "L2 flushed before every timed step (the 19 MB FP4 cache fits in L2)"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import workloads as W
        C = _C()
        B, N = self.B, self.N
        self.kv = torch.empty((B, N, 288), dtype=torch.uint8, device=dev)
        for b in range(B):
            C.csa2_fp4_pack(W.fp4_rows("kv", self.seq0 + b, 0, N, N, dev),
                            C.FP4_E4M3x16, out=self.kv[b])
        self.q = W.normal_tensor((B, 1, self.H, 512), 6001, 0, torch.bfloat16, dev)
        self.swa = W.normal_tensor((B, 128, 512), 6002, 0, torch.bfloat16, dev)
        self.sink = W.normal_tensor((self.H,), 6003, 0, torch.float32, dev)
        self.q_pos = torch.full((B, 1), self.t, dtype=torch.int64, device=dev)
        self.nv = torch.full((B, 1), self.V, dtype=torch.int64, device=dev)
        # decode compressor: the block's first 127 tokens are in the state, the step brings the 128th
        m = self.m
        pre_c = W.normal_tensor((B, m - 1, 512), 6004, 0, torch.bfloat16, dev)
        pre_z = W.normal_tensor((B, m - 1, 512), 6005, 0, torch.bfloat16, dev)
        self.state = C.csa2_compress_state(B, 512, m, torch.bfloat16, dev, overlap=False)
        C.csa2_compress_state_seed(pre_c, pre_z, m, self.state)
        self.c_new = W.normal_tensor((B, 512), 6006, 0, torch.bfloat16, dev)
        self.z_new = W.normal_tensor((B, 512), 6007, 0, torch.bfloat16, dev)
        self.pos_new = torch.full((B,), self.t, dtype=torch.int64, device=dev)
        self.out = torch.empty((B, 1, self.H, 512), dtype=torch.bfloat16, device=dev)
        self.ws = C._ws(C.csa2_sparse_attn_workspace_bytes(B, 1, self.H, N, 128, N=N, swa_cap=128), dev)
        self.e2e_in = [self.q, self.c_new, self.z_new]
        self.e2e_out = [self.out]
        torch.cuda.synchronize()

    def write(self):
        C = _C()
        C.csa2_compress_step(self.c_new, self.z_new, self.m, self.pos_new, self.state, flags=C.W_NORM | C.W_ROPE,
                             out=self.kv, out_fmt="fp4", out_seq_stride=self.N)

    def main(self):
        _C().csa2_dense_attn(self.q, self.kv, self.nv, self.N, self.swa, self.q_pos, self.sink, window=128,
                             out=self.out, ws=self.ws)

    def pre(self):
        self.write()

    def launches_per_step(self):
        return 1 + 3              # compress step; query prep, attention, split combine

    def main_amount(self):
        """FLOPs of one attention launch: QK and PV over (V + 128) rows, 64 heads."""
        return self.B * self.H * (self.V + 128) * 512 * 4

    def stages(self):
        B = self.B
        return [("compress step (m' = 128, FP4 row)", self.write, B * (2 * 1024 + 2 * 128 * 1024 + 288), 0),
                ("dense attention", self.main, B * ((self.V) * 288 + 128 * 1024 + self.H * 1024 * 2),
                 self.main_amount())]

    def queries(self):
        return self.B

    def entries(self):
        return self.B * self.V

    def oracle_prepare(self, b=0):
        from compressed_sparse_attention_06_gb300 import workloads as W
        from oracle import csa2_oracle as O
        self.o_kv = O.nvfp4_unpack(O.nvfp4_pack(W.fp4_rows("kv", self.seq0 + b, 0, self.N, self.N, "cpu").numpy()))
        self.o_q = (self.q[b, 0].double().cpu().numpy(), self.swa[b].double().cpu().numpy(),
                    self.sink.double().cpu().numpy())

    def oracle_query(self):
        from oracle import csa2_oracle as O
        q, swa, sink = self.o_q
        return O.dense_attn(q, self.o_kv, swa, 0, self.t, self.m, sink, 128)[0]

    def oracle_sample_text(self, n):
        return (f"{n} query(ies) of sequence 0 (oracle dense attention over {self.V} dequantised FP4 entries + "
                f"128 window rows, 64 heads; numpy f64), {os.uname().machine}")


class CompressStepM4(Workload):
    """The CSA compressor in decode (overlapped, m = 4) for 64 sequences: every step
    stores the new token's rows in the compressor state and, for the token that
    completes a block, writes the FP4 main-KV row and the MXFP4 indexer-key row."""
    name = "compress_step_m4"
    main_name = "csa2_compress_step (overlap m=4, c=512 FP4 row + c=128 MXFP4 row)"
    kernel_files = ("compress.cu", "csa2_internal.cuh")
    flush_l2 = True

    def __init__(self, B=64, N=None, seq0=0):
        self.B, self.m = B, 4
        self.t = 4 * 4096 - 1                 # completes a block at every timed step

    def config(self):
        return {"workload": self.name, "batch": self.B, "m": self.m, "overlap": True,
                "rows": "main KV c=512 -> FP4 288 B; indexer K c=128 -> MXFP4 68 B", "flags": "RMSNorm + RoPE",
                "l2": "L2 flushed before every timed step (state and rows fit in L2)"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import workloads as W
        C = _C()
        B, m = self.B, self.m
        self.new = {c: [W.normal_tensor((B, c), 6100 + c, k, torch.bfloat16, dev) for k in range(4)]
                    for c in (512, 128)}
        self.bias = {c: (W.normal_tensor((m, c), 6200 + c, 0, torch.float32, dev, std=0.1),
                         W.normal_tensor((m, c), 6200 + c, 1, torch.float32, dev, std=0.1)) for c in (512, 128)}
        self.state = {}
        for c in (512, 128):
            self.state[c] = C.csa2_compress_state(B, c, m, torch.bfloat16, dev)
            pre = [W.normal_tensor((B, 2 * m - 1, c), 6300 + c, k, torch.bfloat16, dev) for k in range(4)]
            C.csa2_compress_state_seed(pre[0], pre[1], m, self.state[c], cb=pre[2], zb=pre[3])
        self.kv = torch.empty((B, 4096, 288), dtype=torch.uint8, device=dev)
        self.ki = torch.empty((B, 4096, 68), dtype=torch.uint8, device=dev)
        self.pos = torch.full((B,), self.t, dtype=torch.int64, device=dev)
        self.e2e_in = self.new[512] + self.new[128]
        self.e2e_out = [self.kv[:, -1].contiguous()]
        torch.cuda.synchronize()

    def step_kv(self):
        C = _C()
        a = self.new[512]
        C.csa2_compress_step(a[0], a[1], self.m, self.pos, self.state[512], cb=a[2], zb=a[3], ba=self.bias[512][0],
                             bb=self.bias[512][1], flags=C.W_NORM | C.W_ROPE, out=self.kv, out_fmt="fp4",
                             out_seq_stride=4096)

    def step_ki(self):
        C = _C()
        a = self.new[128]
        C.csa2_compress_step(a[0], a[1], self.m, self.pos, self.state[128], cb=a[2], zb=a[3], ba=self.bias[128][0],
                             bb=self.bias[128][1], flags=C.W_NORM | C.W_ROPE, out=self.ki, out_fmt="mxfp4",
                             out_seq_stride=4096)

    def main(self):
        self.step_kv()

    def post(self):
        self.step_ki()

    def launches_per_step(self):
        return 2

    def main_amount(self):
        """Bytes of one main-KV step: the token's four rows in, the block's 4 x 4 state
        rows read and 2 x 4 written back, the FP4 row out."""
        return self.B * (4 * 1024 + 16 * 1024 + 8 * 1024 + 288)

    def stages(self):
        return [("compress step, main KV (FP4)", self.step_kv, self.main_amount(), 0),
                ("compress step, indexer K (MXFP4)", self.step_ki, self.B * (4 * 256 + 24 * 256 + 68), 0)]

    def queries(self):
        return self.B

    def entries(self):
        return self.B


class PrefillVarlenCompress(Workload):
    """Packed-sample prefill write path: 32 samples of 1,000 .. 4,000 tokens back to
    back (cu_tokens offsets), overlapped compressor m = 4, each sample compressed alone
    into its own cache rows: FP4 main KV (c = 512) and MXFP4 indexer keys (c = 128)."""
    name = "prefill_varlen_compress"
    main_name = "csa2_compress_varlen (overlap m=4, c=512 -> FP4 rows)"
    kernel_files = ("compress.cu", "csa2_internal.cuh")

    def __init__(self, B=32, N=None, seq0=0):
        self.S, self.m = B, 4

    def config(self):
        return {"workload": self.name, "samples": self.S, "tokens": self.T, "m": self.m, "overlap": True,
                "rows": "main KV c=512 -> FP4 288 B; indexer K c=128 -> MXFP4 68 B", "flags": "RMSNorm + RoPE",
                "l2": f"inputs larger than L2 ({self.T * (4 * 512 + 4 * 128) * 2 / 1e6:.0f} MB of token rows)"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import workloads as W
        C = _C()
        u = W.uniform(self.S, 6401, 0, "cpu")
        self.lens = [int(1000 + 3000 * float(x)) for x in u]
        self.T, self.maxlen = sum(self.lens), max(self.lens)
        self.cu = torch.tensor([0] + list(np.cumsum(self.lens)), dtype=torch.int64, device=dev)
        self.rows = {c: [W.normal_tensor((self.T, c), 6410 + c, k, torch.bfloat16, dev) for k in range(4)]
                     for c in (512, 128)}
        self.bias = {c: (W.normal_tensor((4, c), 6420 + c, 0, torch.float32, dev, std=0.1),
                         W.normal_tensor((4, c), 6420 + c, 1, torch.float32, dev, std=0.1)) for c in (512, 128)}
        ne = self.maxlen // self.m
        self.kv = torch.empty((self.S, ne, 288), dtype=torch.uint8, device=dev)
        self.ki = torch.empty((self.S, ne, 68), dtype=torch.uint8, device=dev)
        self.entries_total = sum(n // self.m for n in self.lens)
        self.e2e_in = self.rows[512] + self.rows[128]
        self.e2e_out = [self.kv]
        torch.cuda.synchronize()

    def write(self, c):
        C = _C()
        a = self.rows[c]
        C.csa2_compress_varlen(a[0], a[1], self.m, self.cu, self.maxlen, cb=a[2], zb=a[3], ba=self.bias[c][0],
                               bb=self.bias[c][1], flags=C.W_NORM | C.W_ROPE, out_fmt="fp4" if c == 512 else "mxfp4",
                               out=self.kv if c == 512 else self.ki)

    def main(self):
        self.write(512)

    def post(self):
        self.write(128)

    def launches_per_step(self):
        return 2

    def main_amount(self):
        """Bytes of the main-KV launch: four bf16 token rows in (each read once: a
        block's rows and, for the next block, its overlap half), FP4 rows out."""
        return self.T * 4 * 1024 + self.entries_total * 288

    def stages(self):
        return [("compress varlen, main KV (FP4)", self.main, self.main_amount(), 0),
                ("compress varlen, indexer K (MXFP4)", self.post, self.T * 4 * 256 + self.entries_total * 68, 0)]

    def queries(self):
        return self.T

    def entries(self):
        return self.entries_total


class PrefillChunk(Workload):
    """Encoder prefill chunk: 8192 queries on a 131,072-token context (m=4 overlap)."""
    name = "prefill_chunk_bf16"
    main_name = "csa2_index_score (bf16 causal scan, 4 queries per key tile)"
    main_bound = "tensor"

    def __init__(self, n_new=8192, seq0=0, N=None):
        self.n_new = n_new

    def config(self):
        return {"workload": self.name, "batch": 1, "queries": self.n_new, "context_tokens": 131072, "m": 4,
                "entries": self.N, "indexer_heads": 64, "heads": 64, "topk": 512, "window": 128,
                "compressor": "overlapped, carried previous-block state",
                "l2": "scores (1.1 GB) and queries larger than L2"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import pipeline as P
        from compressed_sparse_attention_06_gb300 import workloads as W
        wl = W.prefill_chunk_bf16(dev, n_new=self.n_new)
        self.wl = wl
        self.N, self.Q, self.m = wl.N, wl.Q, wl.m
        self.nce = wl.meta["n_ctx_entries"]
        self.kv = torch.empty((1, self.N, 512), dtype=torch.bfloat16, device=dev)
        self.kv[0, :self.nce] = wl["kv_ctx"][0]
        self.pos0 = torch.tensor([wl.meta["pos0"]], dtype=torch.int64, device=dev)
        self.buf = P.alloc_prefill(self.Q, self.N, 64, 512, dev, wl.q_pos, self.m, swa_cap=wl.meta["swa_cap"])
        self.V_sum = int(self.buf.n_visible.sum())
        self.e2e_in = [wl["Ca"], wl["Cb"], wl["Za"], wl["Zb"], wl["qI"], wl["w"], wl["q"]]
        self.e2e_out = [self.buf.out, self.buf.idx]

    def compress(self):
        C = _C()
        wl = self.wl
        C.csa2_compress(wl["Ca"], wl["Za"], self.m, cb=wl["Cb"], zb=wl["Zb"], ba=wl["Ba"], bb=wl["Bb"],
                        prev_cb=wl["prev_Cb"], prev_zb=wl["prev_Zb"], pos0=self.pos0, flags=C.W_NORM | C.W_ROPE,
                        out=self.kv[0, self.nce:], out_seq_stride=0)

    def main(self):
        wl = self.wl
        _C().csa2_index_score(wl["qI"], wl["w"], wl["KI"], self.buf.n_visible, scores=self.buf.scores)

    def topk(self):
        _C().csa2_topk(self.buf.scores, self.buf.n_visible, 512, out_idx=self.buf.idx, ws=self.buf.topk_ws)

    def attn(self):
        wl = self.wl
        _C().csa2_sparse_attn(wl["q"], self.kv, self.buf.idx, wl["swa"], wl.q_pos, wl["sink"],
                              swa_pos0=wl.meta["swa_pos0"], out=self.buf.out, ws=self.buf.attn_ws)

    def pre(self):
        self.compress()

    def post(self):
        self.topk(); self.attn()

    def launches_per_step(self):
        return 4

    def main_amount(self):
        return 2 * self.V_sum * 64 * 128          # flops of the causal indexer contraction

    def stages(self):
        Q = self.Q
        return [("compress (overlap, m=4)", self.compress, self.n_new * 512 * 2 * 4 + 2048 * 1024, 0),
                ("index scan", self.main, self.N * 256 + Q * 64 * 260 + Q * self.N * 4, self.main_amount()),
                ("top-512", self.topk, Q * self.N * 4, 0),
                ("sparse attention", self.attn, Q * (640 * 1024 + 64 * 512 * 4), Q * 64 * 640 * 512 * 4)]

    def queries(self):
        return self.Q

    def entries(self):
        return self.V_sum


class TinyLayer(Workload):
    """Tiny fp32 Full layer (CUDA-core path)."""
    name = "tiny_full_layer_fp32"
    main_name = "csa2_index_score (fp32, CUDA cores)"
    dtype = "fp32"

    def __init__(self, seq0=0, N=None):
        pass

    def config(self):
        return {"workload": self.name, "tokens": 4096, "m": 2, "entries": 2048, "indexer_heads": 8, "heads": 16,
                "queries": 4, "l2": "inputs fit in L2 (correctness workload)"}

    def setup(self, dev):
        from compressed_sparse_attention_06_gb300 import pipeline as P
        from compressed_sparse_attention_06_gb300 import workloads as W
        wl = W.tiny_full_layer(dev)
        self.wl = wl
        self.kv = torch.empty((1, 2048, 512), dtype=torch.float32, device=dev)
        self.nv = P.visible_entries(wl.q_pos, wl.m)
        self.scores = torch.empty((1, 4, 2048), dtype=torch.float32, device=dev)
        self.idx = torch.empty((1, 4, 512), dtype=torch.int32, device=dev)
        self.out = torch.empty((1, 4, 16, 512), dtype=torch.float32, device=dev)
        self.e2e_in = [wl["qI"], wl["w"], wl["q"]]
        self.e2e_out = [self.out, self.idx]

    def compress(self):
        C = _C()
        wl = self.wl
        C.csa2_compress(wl["Ca"], wl["Za"], wl.m, ba=wl["Ba"], flags=C.W_NORM | C.W_ROPE, out=self.kv[0])

    def main(self):
        wl = self.wl
        _C().csa2_index_score(wl["qI"], wl["w"], wl["KI"], self.nv, scores=self.scores)

    def post(self):
        wl = self.wl
        _C().csa2_topk(self.scores, self.nv, 512, out_idx=self.idx)
        _C().csa2_sparse_attn(wl["q"], self.kv, self.idx, wl["swa"], wl.q_pos, wl["sink"], out=self.out)

    def pre(self):
        self.compress()

    def launches_per_step(self):
        return 5

    def main_amount(self):
        return 2048 * 128 * 4 * 4

    def stages(self):
        return [("compress", self.compress, 4096 * 512 * 8 + 2048 * 2048, 0),
                ("index scan", self.main, self.main_amount(), 0)]

    def queries(self):
        return 4

    def entries(self):
        return int(self.nv.sum())


class _RowMap:
    """Indexable view over a dict of gathered rows (the oracle indexes kv[s])."""

    def __init__(self, rows):
        self.rows = rows

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


WORKLOADS = {c.name: c for c in (FP4Decode, DecodeBF16, ReindexReuse, PrefillChunk, TinyLayer, HCADecode,
                                  CompressStepM4, V4ProDecode, PrefillVarlenCompress)}


def _make(args, seq0=0):
    kw = {"seq0": seq0}
    if args.n_ctx:
        kw["N"] = args.n_ctx
    if args.n_new:
        if args.workload != "prefill_chunk_bf16":
            raise SystemExit("--n-new applies to prefill_chunk_bf16 only")
        kw["n_new"] = args.n_new
    return WORKLOADS[args.workload](**kw)


# ----------------------------------------------------------------------------- arms
def _time_stages(wl, stream, reps):
    """Each stage alone, `reps` times, CUDA events around every launch (median).
    A GPU spin of about a millisecond is queued before each timed stage, so the
    stage's launches are already queued when its start event runs: the interval is
    GPU time, not host launch overhead."""
    hbm, bf16, _, _ = _peaks()
    out = {}
    for st in wl.stages():
        name, fn, nbytes, flops = st[:4]
        kind = st[4] if len(st) > 4 else "bf16"
        fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a, b in evs:
            torch.cuda._sleep(2_000_000)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ms = sorted(a.elapsed_time(b) for a, b in evs)[reps // 2]
        d = {"ms": ms, "GB_per_s": nbytes / (ms * 1e-3) / 1e9, "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm}
        if flops:
            d["TFLOP_per_s"] = flops / (ms * 1e-3) / 1e12
            # a kind::mxf4 MMA runs at the FP4 rate: the measured bf16 peak times the
            # nominal dense FP4 / bf16 ratio (13.5 / 2.25 PFLOP/s)
            peak = bf16 * FP4_PER_BF16 if kind == "fp4" else bf16
            d["tensor_frac"] = d["TFLOP_per_s"] / peak
            d["tensor_peak"] = {"TFLOP_per_s": peak, "dtype": kind}
        out[name] = d
    return out


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
    C = _C()
    C.load()
    wl = _make(args, seq0=rank * 8)
    wl.setup(dev)
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(dev)
    clocks.start()

    # the step's side work (cache rows for later steps) forks onto a second stream after
    # the scan (beside the selections and the attention, which leave SMs free) and joins
    # at the end of the step
    side_stream = torch.cuda.Stream(dev) if wl.has_side else None
    g_side = None

    def fork_side():
        if side_stream is None:
            return
        side_stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side_stream):
            if g_side is not None:
                g_side.replay()
            else:
                wl.side()

    def join_side():
        if side_stream is not None:
            torch.cuda.current_stream(dev).wait_stream(side_stream)

    # warm-up (also sets kernel attributes before any graph capture)
    for _ in range(max(1, args.warmup)):
        wl.pre(); wl.main(); fork_side(); wl.post(); join_side()
    C.csa2_ctx_check()
    g_pre = g_post = None
    if not args.no_graph:
        g_pre, g_post = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g_pre, stream=s):
                wl.pre()
            with torch.cuda.graph(g_post, stream=s):
                wl.post()
            if side_stream is not None:
                g_side_new = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_side_new, stream=s):
                    wl.side()
        stream.wait_stream(s)
        if side_stream is not None:
            g_side = g_side_new
        for _ in range(2):
            g_pre.replay(); wl.main(); fork_side(); g_post.replay(); join_side()
    torch.cuda.synchronize()

    def step(ev0=None, ev1=None):
        if g_pre is not None:
            g_pre.replay()
        else:
            wl.pre()
        if ev0 is not None:
            ev0.record(stream)
        wl.main()
        if ev1 is not None:
            ev1.record(stream)
        fork_side()
        if g_post is not None:
            g_post.replay()
        else:
            wl.post()
        join_side()

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # workloads whose data fit in L2 flush it before every step (a 256 MB write, outside
    # the step's own event interval); the others stream more than L2 per step
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if wl.flush_l2 else None
    sevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)] \
        if flush is not None else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        if flush is not None:
            flush.zero_()
            sevs[i][0].record(stream)
        step(*evs[i])
        if flush is not None:
            sevs[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    C.csa2_ctx_check()
    ms_total = t0.elapsed_time(t1) if flush is None else sum(a.elapsed_time(b) for a, b in sevs)
    main_ms = sum(a.elapsed_time(b) for a, b in evs) / K
    if dist is not None:
        tt = torch.tensor([ms_total, main_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_total, main_ms = float(tt[0]), float(tt[1])
    ms_step = ms_total / K

    stages = _time_stages(wl, stream, max(5, K))
    C.csa2_ctx_check()

    # end to end: host inputs -> device, step, result -> host, every step.  With graphs
    # on, one CUDA graph holds the whole step -- the copies from and to pinned host
    # memory included, so every replay moves the step's bytes -- and the host waits for
    # each step's result before the next, as a decode loop does.
    h2d, d2h = wl.e2e_inputs()
    torch.cuda.synchronize()

    def e2e_step():
        wl.e2e_copy_in()
        wl.pre()
        wl.main()
        fork_side()
        wl.post()
        join_side()
        wl.e2e_copy_out()

    g_e2e = None
    g_side = None                          # the one e2e graph captures the side branch itself
    if not args.no_graph:
        g_e2e = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g_e2e, stream=s):
                e2e_step()
        stream.wait_stream(s)
    run_e2e = g_e2e.replay if g_e2e is not None else e2e_step
    for _ in range(2):
        run_e2e(); torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = time.perf_counter()
    for _ in range(K):
        run_e2e()
        torch.cuda.synchronize()
    e_s = time.perf_counter() - e0
    if dist is not None:
        tt = torch.tensor([e_s], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e_s = float(tt[0])

    hbm, bf16, bf16s, src = _peaks()
    if wl.main_bound == "hbm":
        achieved = wl.main_amount() / (main_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "bytes_per_launch": wl.main_amount()}
    else:
        achieved = wl.main_amount() / (main_ms * 1e-3) / 1e12
        peak = bf16s if ms_step > 5.0 else bf16
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "flops_per_launch": wl.main_amount()}
    traffic = _profile_traffic(wl.profile, _kernel_hash(wl.kernel_files)) if wl.profile else None
    roof.update({"traffic": traffic, "kernel": wl.main_name, "kernel_ms": main_ms, "peak_source": src})
    value = world * wl.queries() / (ms_step * 1e-3)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic (seeded counter-based generator)",
        "config": {**wl.config(), "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "cuda_graph": g_pre is not None},
        "entries_per_s": world * wl.entries() / (ms_step * 1e-3),
        "roofline": roof,
        "stages": stages,
        "e2e": {"value": world * wl.queries() * K / e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "one_graph_per_step": g_e2e is not None},
        "gpu_launches": wl.launches_per_step() * K,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline and hasattr(wl, "oracle_query"):
        res["cpu_baseline"] = cpu_baseline(wl, args)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def cpu_baseline(wl, args):
    """The oracle, as it stands, on a bounded sample of the same workload."""
    wl.oracle_prepare(0)
    n = args.cpu_queries
    t0 = time.perf_counter()
    for _ in range(n):
        wl.oracle_query()
    dt = time.perf_counter() - t0
    cores = wl.oracle_cores() if hasattr(wl, "oracle_cores") else _cores()
    return {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": wl.oracle_sample_text(n)}


def run_reference(args):
    rank, world, _ = _env_rank()
    if rank != 0:
        return
    wl = _make(args)
    if not hasattr(wl, "oracle_query"):
        print(json.dumps({"impl": "reference", "unavailable": f"no oracle sample defined for {wl.name}"}))
        return
    wl.oracle_prepare(0)
    for _ in range(args.warmup):
        wl.oracle_query()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        wl.oracle_query()
    dt = time.perf_counter() - t0
    v = args.steps / dt
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
           "config": wl.config(),
           "cpu_baseline": {"value": v, "unit": UNIT,
                            "cores": wl.oracle_cores() if hasattr(wl, "oracle_cores") else _cores(),
                            "kind": "oracle", "sample": "each step = " + wl.oracle_sample_text(1)},
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
    ap.add_argument("--n-new", type=int, default=None,
                    help="prefill_chunk_bf16: queries of the chunk (default 8192; smaller for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
