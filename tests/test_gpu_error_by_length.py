"""Error of the Full decode step against the oracle as a function of context length
(DSA-to-CSA/HCA page, «数值与 kernel»: each precision path against a high-precision
reference, reported by sequence length), for the FP4-cache path (MXFP4 indexer
keys and query, FP4 main KV) and the bf16 path, at 4K, 64K, 256K and 1M entries.

Two errors per point:
  * kernel error -- the step against the oracle on the same quantised inputs: the
    scores (relative to their rms), the top-512 (exact up to the tie window) and
    the attention output (the parity rule, 2e-2 for a bf16 output path).  Asserted.
  * format error -- the same step against the oracle on the unquantised inputs (f32
    rows): with the step's own selection (what the row format costs the attention)
    and with the oracle's own selection on unquantised scores (what the format costs
    the whole layer, selection changes included), as relative L2 errors, plus the
    overlap of the two selections.  Reported, not asserted (a property of the format).
With CSA2_ERROR_REPORT set, each point is appended to that file as a JSON line."""
import json
import os

import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import pipeline as P
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np, topk_swaps

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENGTHS = [4096, 65536, 262144, 1 << 20]
CHUNK = 1 << 18


def _rel(g, o):
    """max |g - o| / (|o| + rms(o)): the parity rule's measure."""
    g, o = np.asarray(g, dtype=np.float64), np.asarray(o, dtype=np.float64)
    return float(np.max(np.abs(g - o) / (np.abs(o) + np.sqrt(np.mean(o ** 2)))))


def _l2(g, o):
    """||g - o|| / ||o|| over every head and dimension."""
    g, o = np.asarray(g, dtype=np.float64), np.asarray(o, dtype=np.float64)
    return float(np.linalg.norm(g - o) / np.linalg.norm(o))


def _oracle_scores(qI, w, rows_f32, V, fmt):
    """Scores of all N entries, the key rows dequantised (fmt 'fp4': MXFP4 packed on
    the host; 'bf16': rounded to bf16; 'f32': as drawn), in chunks of rows."""
    N = rows_f32.shape[0]
    out = np.full(N, -np.inf)
    for r0 in range(0, V, CHUNK):
        r1 = min(V, r0 + CHUNK)
        x = rows_f32[r0:r1]
        if fmt == "fp4":
            K = O.mxfp4_unpack(O.mxfp4_pack(x.numpy()))
        elif fmt == "bf16":
            K = x.to(torch.bfloat16).double().numpy()
        else:
            K = x.double().numpy()
        out[r0:r1] = O.index_score(qI, w, K, r1 - r0)[: r1 - r0]
    return out


def _rows(kv_f32, ids, fmt):
    x = kv_f32[torch.as_tensor(ids, dtype=torch.int64)]
    if fmt == "fp4":
        v = O.nvfp4_unpack(O.nvfp4_pack(x.numpy()))
    elif fmt == "bf16":
        v = x.to(torch.bfloat16).double().numpy()
    else:
        v = x.double().numpy()
    return {int(i): v[j] for j, i in enumerate(ids)}


@pytest.mark.parametrize("path", ["fp4", "bf16"])
@pytest.mark.parametrize("N", LENGTHS, ids=[f"{n // 1024}K" for n in LENGTHS])
def test_error_by_context_length(path, N):
    wl = W.fp4_decode(DEV, B=1, N=N)
    t = wl.tensors
    ki_f = W.fp4_rows("KI", 0, 0, N, N, DEV)
    kv_f = W.fp4_rows("kv", 0, 0, N, N, DEV)
    if path == "fp4":
        kI = C.csa2_fp4_pack(ki_f.view(1, N, 128), C.MXFP4_E8M0x32)
        kv = C.csa2_fp4_pack(kv_f.view(1, N, 512), C.FP4_E4M3x16)
    else:
        kI = ki_f.to(torch.bfloat16).view(1, N, 128)
        kv = kv_f.to(torch.bfloat16).view(1, N, 512)
    q_pos = wl.q_pos
    nv = P.visible_entries(q_pos, 1)
    V = int(nv[0, 0])
    buf = P.alloc_decode(1, 1, N, 64, 512, DEV, out_dtype=torch.float32)
    P.full_decode_step(t["qI"], t["w"], kI, t["q"], kv, t["swa"], q_pos, nv, t["sink"], buf)
    C.csa2_ctx_check()

    ki_h, kv_h = ki_f.cpu(), kv_f.cpu()
    qI_bf = t["qI"][0, 0].float().cpu().numpy()
    w = t["w"][0, 0].double().cpu().numpy()
    q = t["q"][0, 0].double().cpu().numpy()
    swa = t["swa"][0].double().cpu().numpy()
    sink = t["sink"].double().cpu().numpy()
    tpos = int(q_pos[0, 0])
    # the oracle on the step's own (quantised) inputs
    qI = O.mxfp4_unpack(O.mxfp4_pack(qI_bf)) if path == "fp4" else qI_bf.astype(np.float64)
    sc = _oracle_scores(qI, w, ki_h, V, path)
    g_sc = to_np(buf.scores[0, 0])
    rms = float(np.sqrt(np.mean(sc[:V] ** 2)))
    score_err = float(np.max(np.abs(g_sc[:V] - sc[:V]))) / rms
    assert score_err <= 1e-5, f"scores off by {score_err:.2e} of their rms"
    g_idx = to_np(buf.idx[0, 0]).astype(np.int64)
    swaps = topk_swaps(g_idx, sc, V, 512)
    pool = O.block_pool(O.block_max(sc, V, 8), V, 8, 2048)
    assert np.array_equal(O.reindex_topk(sc, pool, V, 512), O.topk(sc, V, 512))   # the pool lemma
    o_ref, lse_ref, _ = O.sparse_attn(q, _rows(kv_h, g_idx[g_idx >= 0], path), g_idx, swa, 0, tpos, sink, 128)
    g_out = to_np(buf.out[0, 0])
    kernel_err = _rel(g_out, o_ref)
    assert_close(g_out, o_ref, 2e-2, f"{path} {N}: attention")
    # the oracle on unquantised inputs: what the storage format costs
    o_same, _, _ = O.sparse_attn(q, _rows(kv_h, g_idx[g_idx >= 0], "f32"), g_idx, swa, 0, tpos, sink, 128)
    sc_f = _oracle_scores(qI_bf.astype(np.float64), w, ki_h, V, "f32")
    idx_f = O.topk(sc_f, V, 512)
    o_f, _, _ = O.sparse_attn(q, _rows(kv_h, idx_f[idx_f >= 0], "f32"), idx_f, swa, 0, tpos, sink, 128)
    overlap = len(set(g_idx.tolist()) & set(idx_f.tolist())) / 512.0
    rec = dict(path=path, N=N, visible=V, score_err_rel_rms=score_err, topk_tie_swaps=swaps,
               attn_kernel_err_max=kernel_err, attn_kernel_err_l2=_l2(g_out, o_ref),
               attn_format_err_l2_same_selection=_l2(g_out, o_same), attn_format_err_l2=_l2(g_out, o_f),
               topk_overlap_with_f32=overlap, score_format_err_rel_rms=float(np.max(np.abs(sc[:V] - sc_f[:V]))) / rms)
    print(json.dumps(rec))
    path_out = os.environ.get("CSA2_ERROR_REPORT")
    if path_out:
        with open(path_out, "a") as f:
            f.write(json.dumps(rec) + "\n")
