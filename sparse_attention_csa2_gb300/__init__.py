"""Python binding of libcsa2.so, the C ABI of the CSA2 attention step on sm_103a.

Argument marshalling only: every step runs in the library's CUDA kernels.  Tensors are
torch CUDA tensors; outputs and workspaces are allocated here with torch and passed as
device pointers; calls are queued on torch's current CUDA stream.  The library must be
built (``python sparse_attention_csa2_gb300/_build.py``); importing this package without
it raises immediately - there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libcsa2.so")

# ------------------------------------------------------------------ constants (csa2.h)
OK, EINVAL, EUNSUPPORTED, ECUDA, ETIMEOUT, EWORKSPACE, EDEVICE_INDEX = range(7)
BF16, FP8_E4M3_ROWSCALE, FP4_E2M1_G32, FP4_E2M1_G16, MXFP4 = range(5)
MODE_FULL, MODE_FULL_POOL, MODE_REINDEX, MODE_REUSE = range(4)
IDX_HEADS, IDX_DIM, HEADS, HEAD_DIM, ROPE_DIM, MAX_TOPK = 32, 128, 64, 512, 64, 1024
MODES = {"full": MODE_FULL, "full_pool": MODE_FULL_POOL, "reindex": MODE_REINDEX, "reuse": MODE_REUSE}


class CSA2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_lib.csa2_status_string(status).decode()} (status {status})")
        self.status = status


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libcsa2.so is not built ({_LIB_PATH}); run python sparse_attention_csa2_gb300/_build.py")
_lib = C.CDLL(_LIB_PATH)
LIB_PATH = _LIB_PATH

_vp, _i32, _i64, _f32, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t


class IndexArgs(C.Structure):
    _fields_ = [("q_idx", _vp), ("w", _vp), ("k_idx", _vp), ("k_scale", _vp), ("k_dtype", _i32),
                ("n_rows", _i32), ("n_seq", _i32), ("n_records", _i64), ("seq_of_row", _vp),
                ("n_visible", _vp), ("cand", _vp), ("n_cand", _vp), ("L", _i64), ("scores", _vp),
                ("block_max", _vp), ("block_size", _i32)]


class TopkArgs(C.Structure):
    _fields_ = [("scores", _vp), ("cand", _vp), ("n_valid", _vp), ("n_rows", _i32), ("L", _i64),
                ("K", _i32), ("idx", _vp), ("workspace", _vp), ("workspace_bytes", _sz)]


class BlockPoolArgs(C.Structure):
    _fields_ = [("block_max", _vp), ("n_visible", _vp), ("n_rows", _i32), ("n_blocks", _i32),
                ("block_size", _i32), ("n_keep", _i32), ("pool", _vp), ("n_pool", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz)]


class AttnArgs(C.Structure):
    _fields_ = [("q", _vp), ("q_pos", _vp), ("seq_of_row", _vp), ("n_rows", _i32), ("n_seq", _i32),
                ("n_records", _i64), ("latents", _vp), ("lat_scale", _vp), ("lat_dtype", _i32),
                ("idx", _vp), ("K", _i32), ("swa", _vp), ("swa_scale", _vp), ("swa_dtype", _i32),
                ("swa_rows", _i64), ("swa_pos0", _vp), ("window", _i32), ("sink", _vp),
                ("rope_theta", _f32), ("softmax_scale", _f32), ("out", _vp), ("sink_mass", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz), ("dev_status", _vp), ("out_bf16", _i32)]


class DecodeArgs(C.Structure):
    _fields_ = [("mode", _i32), ("index", IndexArgs), ("K", _i32), ("block_size", _i32),
                ("n_keep", _i32), ("pool_len", _i32), ("pool", _vp), ("n_pool", _vp), ("idx", _vp),
                ("attn", AttnArgs), ("workspace", _vp), ("workspace_bytes", _sz),
                ("stage_events", _vp * 4)]


class ShardArgs(C.Structure):
    _fields_ = [("scores", _vp), ("n_valid", _vp), ("n_rows", _i32), ("L", _i64), ("K", _i32),
                ("first_record", _i64), ("out_scores", _vp), ("out_pos", _vp), ("out_cnt", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz)]


class MergeArgs(C.Structure):
    _fields_ = [("scores", _vp), ("pos", _vp), ("cnt", _vp), ("n_rows", _i32), ("n_lists", _i32),
                ("K_in", _i32), ("K", _i32), ("idx", _vp), ("workspace", _vp), ("workspace_bytes", _sz)]


class PartialArgs(C.Structure):
    _fields_ = [("attn", AttnArgs), ("part_o", _vp), ("part_ml", _vp), ("range_first", _i64),
                ("range_count", _i64), ("skip_window", _i32)]


class AttnMergeArgs(C.Structure):
    _fields_ = [("part_o", _vp), ("part_ml", _vp), ("n_parts", _i32), ("part_tiles", _i32), ("n_rows", _i32),
                ("q_pos", _vp), ("sink", _vp), ("rope_theta", _f32), ("out", _vp), ("out_bf16", _i32),
                ("sink_mass", _vp)]


class WriteArgs(C.Structure):
    _fields_ = [("n_rows", _i64), ("x", _vp), ("x_f32", _i32), ("pos", _vp), ("rope_theta", _f32),
                ("dst_row", _vp), ("cache_rows", _i64), ("out_dtype", _i32), ("codes", _vp), ("scales", _vp),
                ("dev_status", _vp)]


class CompressArgs(C.Structure):
    _fields_ = [("n_entries", _i64), ("ratio", _i32), ("kv", _vp), ("gate", _vp), ("x_f32", _i32), ("out", _vp)]


class QueryProjArgs(C.Structure):
    _fields_ = [("n_tokens", _i32), ("hidden", _i32), ("q_rank", _i32), ("n_heads", _i32), ("x", _vp),
                ("w_dq", _vp), ("g_q", _vp), ("w_uq", _vp), ("g_head", _vp), ("eps", _f32), ("q", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz), ("dev_status", _vp)]


class ExpandArgs(C.Structure):
    _fields_ = [("n_records", _i64), ("codes", _vp), ("exps", _vp), ("out", _vp)]


class LinearArgs(C.Structure):
    _fields_ = [("n_tokens", _i32), ("in_features", _i32), ("out_features", _i32), ("x", _vp), ("w", _vp),
                ("out", _vp), ("dev_status", _vp)]


class OutProjArgs(C.Structure):
    _fields_ = [("n_tokens", _i32), ("n_heads", _i32), ("n_groups", _i32), ("o_rank", _i32), ("hidden", _i32),
                ("o", _vp), ("w_oa", _vp), ("w_ob", _vp), ("out", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz), ("dev_status", _vp)]


def _sig(name, argtypes, restype):
    f = getattr(_lib, name)
    f.argtypes = argtypes
    f.restype = restype
    return f


_lib.csa2_status_string.argtypes = [C.c_int]
_lib.csa2_status_string.restype = C.c_char_p
_index_scores = _sig("csa2_index_scores", [C.POINTER(IndexArgs), _vp], C.c_int)
_topk_ws = _sig("csa2_topk_workspace_size", [C.POINTER(TopkArgs)], _sz)
_topk = _sig("csa2_topk", [C.POINTER(TopkArgs), _vp], C.c_int)
_pool_ws = _sig("csa2_block_pool_workspace_size", [C.POINTER(BlockPoolArgs)], _sz)
_block_pool = _sig("csa2_block_pool", [C.POINTER(BlockPoolArgs), _vp], C.c_int)
_attn_ws = _sig("csa2_sparse_attn_workspace_size", [C.POINTER(AttnArgs)], _sz)
_sparse_attn = _sig("csa2_sparse_attn", [C.POINTER(AttnArgs), _vp], C.c_int)
_decode_ws = _sig("csa2_fused_decode_workspace_size", [C.POINTER(DecodeArgs)], _sz)
_fused_decode = _sig("csa2_fused_decode", [C.POINTER(DecodeArgs), _vp], C.c_int)
_decode_launches = _sig("csa2_fused_decode_launch_count", [C.POINTER(DecodeArgs)], C.c_int32)
_write_records = _sig("csa2_write_records", [C.POINTER(WriteArgs), _vp], C.c_int)
_compress = _sig("csa2_compress", [C.POINTER(CompressArgs), _vp], C.c_int)
_query_proj = _sig("csa2_query_proj", [C.POINTER(QueryProjArgs), _vp], C.c_int)
_query_proj_ws = _sig("csa2_query_proj_workspace_size", [C.POINTER(QueryProjArgs)], _sz)
_out_proj = _sig("csa2_out_proj", [C.POINTER(OutProjArgs), _vp], C.c_int)
_out_proj_ws = _sig("csa2_out_proj_workspace_size", [C.POINTER(OutProjArgs)], _sz)
_linear = _sig("csa2_linear", [C.POINTER(LinearArgs), _vp], C.c_int)
_expand = _sig("csa2_expand_mxfp4", [C.POINTER(ExpandArgs), _vp], C.c_int)
_version = _sig("csa2_version", [], C.c_int32)
_read_status = _sig("csa2_read_device_status", [_vp, C.POINTER(C.c_int32), _vp], C.c_int)
_set_tuning = _sig("csa2_set_tuning", [C.c_int32, C.c_int32], C.c_int)
_shard_ws = _sig("csa2_shard_candidates_workspace_size", [C.POINTER(ShardArgs)], _sz)
_shard = _sig("csa2_shard_candidates", [C.POINTER(ShardArgs), _vp], C.c_int)
_merge_ws = _sig("csa2_merge_candidates_workspace_size", [C.POINTER(MergeArgs)], _sz)
_merge = _sig("csa2_merge_candidates", [C.POINTER(MergeArgs), _vp], C.c_int)
_partial_tiles = _sig("csa2_attn_partial_tiles", [C.c_int32, C.c_int32], C.c_int32)
_partial = _sig("csa2_sparse_attn_partial", [C.POINTER(PartialArgs), _vp], C.c_int)
_attn_merge = _sig("csa2_attn_merge", [C.POINTER(AttnMergeArgs), _vp], C.c_int)
_selftest_wait = _sig("csa2_selftest_wait_timeout", [_vp, C.c_int32, _vp], C.c_int)

# launch-heuristic overrides (csa2_tuning)
TUNE_SCAN_SEGMENTS, TUNE_SCAN_WARP_MMA, TUNE_SCAN_CLUSTER, TUNE_PROJ_KSPLIT, TUNE_ATTN_ROWS = 0, 1, 2, 3, 4
_TUNE_DEFAULTS = {TUNE_SCAN_SEGMENTS: 0, TUNE_SCAN_WARP_MMA: 0, TUNE_SCAN_CLUSTER: 1, TUNE_PROJ_KSPLIT: 0,
                  TUNE_ATTN_ROWS: 0}


def version() -> int:
    return int(_version())


def read_device_status(dev_status) -> int:
    """The status word [1] int32 that kernels wrote (csa2_read_device_status: synchronizes
    the current stream)."""
    out = C.c_int32(0)
    _check(_read_status(C.c_void_p(_ptr(dev_status)), C.byref(out), _stream()), "csa2_read_device_status")
    return int(out.value)


def selftest_wait_timeout(dev_status, tries: int = 1000) -> None:
    """Runs the bounded-wait self-test: dev_status (int32 device tensor) receives ETIMEOUT."""
    _check(_selftest_wait(C.c_void_p(_ptr(dev_status)), int(tries), _stream()), "csa2_selftest_wait_timeout")


def set_tuning(knob: int, value: int) -> None:
    """Process-wide override of one launch heuristic (csa2_set_tuning)."""
    _check(_set_tuning(int(knob), int(value)), "csa2_set_tuning")


def reset_tuning() -> None:
    """Every launch heuristic back to automatic."""
    for k, v in _TUNE_DEFAULTS.items():
        set_tuning(k, v)


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _check(status: int, what: str):
    if status != OK:
        raise CSA2Error(status, what)


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t):
    return t.device


def _ws(nbytes: int, device):
    if nbytes == 0:
        return None, 0
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return buf, nbytes


def _key_dtype(k_idx, k_scale):
    if k_idx.element_size() == 2:
        return BF16
    if k_idx.element_size() == 1 and k_scale is not None and k_scale.dtype == torch.uint8:
        if k_idx.shape[-1] != 64 or k_scale.shape[-1] != 4:
            raise ValueError("MXFP4 keys are [..., 64] code bytes with [..., 4] exponent bytes")
        return MXFP4
    if k_idx.element_size() == 1 and k_scale is not None:
        return FP8_E4M3_ROWSCALE
    raise ValueError("indexer keys must be bf16 (2-byte), E4M3 bytes with fp32 row scales, or MXFP4")


def _lat_dtype(lat, lat_scale):
    if lat.element_size() == 2:
        return BF16
    g = HEAD_DIM // lat_scale.shape[-1]
    return FP4_E2M1_G32 if g == 32 else FP4_E2M1_G16


def _i32t(x, device):
    return torch.as_tensor(x, dtype=torch.int32, device=device).contiguous()


def _i64t(x, device):
    return torch.as_tensor(x, dtype=torch.int64, device=device).contiguous()


def _index_args(q_idx, w, k_idx, k_scale, seq_of_row, n_visible, cand=None, n_cand=None):
    a = IndexArgs()
    a.q_idx, a.w, a.k_idx, a.k_scale = _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(k_scale)
    a.k_dtype = _key_dtype(k_idx, k_scale)
    a.n_rows = q_idx.shape[0]
    a.n_seq, a.n_records = k_idx.shape[0], k_idx.shape[1]
    a.seq_of_row, a.n_visible = _ptr(seq_of_row), _ptr(n_visible)
    if cand is not None:
        a.cand, a.n_cand, a.L = _ptr(cand), _ptr(n_cand), cand.shape[1]
    return a


# ------------------------------------------------------------------ public calls
def index_scores(q_idx, w, k_idx, k_scale, seq_of_row, n_visible, cand=None, n_cand=None,
                 block_size: int = 0):
    """Indexer scores [n_rows, L] (fp32, -inf where not a candidate) and, with block_size > 0,
    the block maxima [n_rows, ceil(N / block_size)]."""
    dev = _dev(q_idx)
    a = _index_args(q_idx, w, k_idx, k_scale, seq_of_row, n_visible, cand, n_cand)
    L = cand.shape[1] if cand is not None else k_idx.shape[1]
    scores = torch.empty((a.n_rows, L), dtype=torch.float32, device=dev)
    a.scores = _ptr(scores)
    bmax = None
    if block_size > 0:
        bmax = torch.empty((a.n_rows, (k_idx.shape[1] + block_size - 1) // block_size), dtype=torch.float32,
                           device=dev)
        a.block_max, a.block_size = _ptr(bmax), block_size
    _check(_index_scores(C.byref(a), _stream()), "csa2_index_scores")
    return (scores, bmax) if block_size > 0 else scores


def topk(scores, n_valid, K: int, cand=None):
    """Top-K of each row as an ascending set of positions, -1 padded: [n_rows, K] int32."""
    dev = _dev(scores)
    a = TopkArgs()
    a.scores, a.cand, a.n_valid = _ptr(scores), _ptr(cand), _ptr(n_valid)
    a.n_rows, a.L, a.K = scores.shape[0], scores.shape[1], K
    idx = torch.empty((a.n_rows, K), dtype=torch.int32, device=dev)
    a.idx = _ptr(idx)
    ws, nb = _ws(int(_topk_ws(C.byref(a))), dev)
    a.workspace, a.workspace_bytes = _ptr(ws), nb
    _check(_topk(C.byref(a), _stream()), "csa2_topk")
    return idx


def block_pool(block_max, n_visible, block_size: int, n_keep: int):
    """Hierarchical pool: ([n_rows, n_keep*block_size] ascending positions -1 padded, [n_rows] sizes)."""
    dev = _dev(block_max)
    a = BlockPoolArgs()
    a.block_max, a.n_visible = _ptr(block_max), _ptr(n_visible)
    a.n_rows, a.n_blocks, a.block_size, a.n_keep = block_max.shape[0], block_max.shape[1], block_size, n_keep
    pool = torch.empty((a.n_rows, n_keep * block_size), dtype=torch.int32, device=dev)
    n_pool = torch.empty((a.n_rows,), dtype=torch.int32, device=dev)
    a.pool, a.n_pool = _ptr(pool), _ptr(n_pool)
    ws, nb = _ws(int(_pool_ws(C.byref(a))), dev)
    a.workspace, a.workspace_bytes = _ptr(ws), nb
    _check(_block_pool(C.byref(a), _stream()), "csa2_block_pool")
    return pool, n_pool


def _attn_args(q, q_pos, seq_of_row, latents, lat_scale, idx, K, swa, swa_scale, swa_pos0, window, sink,
               theta, softmax_scale, out, sink_mass):
    a = AttnArgs()
    a.q, a.q_pos, a.seq_of_row = _ptr(q), _ptr(q_pos), _ptr(seq_of_row)
    a.n_rows, a.n_seq, a.n_records = q.shape[0], latents.shape[0], latents.shape[1]
    a.latents, a.lat_scale, a.lat_dtype = _ptr(latents), _ptr(lat_scale), _lat_dtype(latents, lat_scale)
    a.idx, a.K = _ptr(idx), K
    a.swa, a.swa_scale = _ptr(swa), _ptr(swa_scale)
    a.swa_dtype = BF16 if swa.element_size() == 2 else FP8_E4M3_ROWSCALE
    a.swa_rows, a.swa_pos0, a.window = swa.shape[1], _ptr(swa_pos0), window
    a.sink, a.rope_theta, a.softmax_scale = _ptr(sink), float(theta), float(softmax_scale)
    a.out, a.sink_mass = _ptr(out), _ptr(sink_mass)
    a.out_bf16 = 1 if (out is not None and out.dtype == torch.bfloat16) else 0
    return a


def sparse_attn(q, q_pos, seq_of_row, latents, lat_scale, idx, swa, swa_scale, swa_pos0, window: int, sink,
                theta: float = 1e4, softmax_scale: float = HEAD_DIM ** -0.5, out_dtype=torch.float32,
                dev_status=None):
    """Attention output [n_rows, 64, 512] (fp32, or bf16 with out_dtype=torch.bfloat16) and
    sink mass [n_rows, 64].  dev_status: optional int32 device tensor of one element that
    the kernels set to a status code (out-of-range index, timed-out wait)."""
    dev = _dev(q)
    out = torch.empty((q.shape[0], HEADS, HEAD_DIM), dtype=out_dtype, device=dev)
    sm = torch.empty((q.shape[0], HEADS), dtype=torch.float32, device=dev)
    a = _attn_args(q, q_pos, seq_of_row, latents, lat_scale, idx, idx.shape[1], swa, swa_scale, swa_pos0, window,
                   sink, theta, softmax_scale, out, sm)
    a.dev_status = _ptr(dev_status)
    ws, nb = _ws(int(_attn_ws(C.byref(a))), dev)
    a.workspace, a.workspace_bytes = _ptr(ws), nb
    _check(_sparse_attn(C.byref(a), _stream()), "csa2_sparse_attn")
    return out, sm


# ------------------------------------------------------------------ record-range split
def shard_candidates(scores, n_valid, K: int, first_record: int):
    """A record range's exact top-K as a candidate list (csa2_shard_candidates): scores [rows,
    K] (ascending positions, -inf pads), positions [rows, K] (-1 pads) and counts [rows]."""
    dev = _dev(scores)
    rows, L = scores.shape
    out_s = torch.empty((rows, K), dtype=torch.float32, device=dev)
    out_p = torch.empty((rows, K), dtype=torch.int32, device=dev)
    out_c = torch.empty((rows,), dtype=torch.int32, device=dev)
    a = ShardArgs(_ptr(scores), _ptr(n_valid), rows, L, K, int(first_record), _ptr(out_s), _ptr(out_p), _ptr(out_c),
                  None, 0)
    ws, nb = _ws(int(_shard_ws(C.byref(a))), dev)
    a.workspace, a.workspace_bytes = _ptr(ws), nb
    _check(_shard(C.byref(a), _stream()), "csa2_shard_candidates")
    return out_s, out_p, out_c


def merge_candidates(scores, pos, cnt, K: int):
    """The rows' top-K of gathered candidate lists scores / pos [lists, rows, K_in] with counts
    [lists, rows] (csa2_merge_candidates): the ascending set of positions [rows, K]."""
    dev = _dev(scores)
    n_lists, rows, k_in = scores.shape
    idx = torch.empty((rows, K), dtype=torch.int32, device=dev)
    a = MergeArgs(_ptr(scores), _ptr(pos), _ptr(cnt), rows, n_lists, k_in, K, _ptr(idx), None, 0)
    ws, nb = _ws(int(_merge_ws(C.byref(a))), dev)
    a.workspace, a.workspace_bytes = _ptr(ws), nb
    _check(_merge(C.byref(a), _stream()), "csa2_merge_candidates")
    return idx


def attn_partial_tiles(K: int, window: int) -> int:
    return int(_partial_tiles(int(K), int(window)))


def sparse_attn_partial(q, q_pos, seq_of_row, latents, lat_scale, idx, swa, swa_scale, swa_pos0, window: int,
                        theta: float = 1e4, softmax_scale: float = HEAD_DIM ** -0.5, range_first: int = 0,
                        range_count: int = 0, skip_window: bool = False):
    """Attention partials of one range's share (csa2_sparse_attn_partial): part_o [rows, tiles,
    64, 512] and part_ml [rows, tiles, 64, 2].  With range_count > 0, idx holds global positions
    and latents only the records [range_first, range_first + range_count)."""
    dev = _dev(q)
    rows = q.shape[0]
    tiles = attn_partial_tiles(idx.shape[1], window)
    part_o = torch.empty((rows, tiles, HEADS, HEAD_DIM), dtype=torch.float32, device=dev)
    part_ml = torch.empty((rows, tiles, HEADS, 2), dtype=torch.float32, device=dev)
    a = PartialArgs()
    a.attn = _attn_args(q, q_pos, seq_of_row, latents, lat_scale, idx, idx.shape[1], swa, swa_scale, swa_pos0, window,
                        None, theta, softmax_scale, None, None)
    a.part_o, a.part_ml = _ptr(part_o), _ptr(part_ml)
    a.range_first, a.range_count, a.skip_window = int(range_first), int(range_count), 1 if skip_window else 0
    _check(_partial(C.byref(a), _stream()), "csa2_sparse_attn_partial")
    return part_o, part_ml


def attn_merge(part_o, part_ml, q_pos, sink, theta: float = 1e4, out_dtype=torch.float32):
    """The output of stacked partials part_o [parts, rows, tiles, 64, 512] / part_ml [parts,
    rows, tiles, 64, 2] (csa2_attn_merge): out [rows, 64, 512] and sink mass [rows, 64]."""
    dev = _dev(part_o)
    n_parts, rows, tiles = part_o.shape[:3]
    out = torch.empty((rows, HEADS, HEAD_DIM), dtype=out_dtype, device=dev)
    sm = torch.empty((rows, HEADS), dtype=torch.float32, device=dev)
    a = AttnMergeArgs(_ptr(part_o), _ptr(part_ml), n_parts, tiles, rows, _ptr(q_pos), _ptr(sink), float(theta),
                      _ptr(out), 1 if out_dtype == torch.bfloat16 else 0, _ptr(sm))
    _check(_attn_merge(C.byref(a), _stream()), "csa2_attn_merge")
    return out, sm


def write_records(x, dst_row, codes, scales, out_dtype: int, pos=None, theta: float = 10000.0, dev_status=None):
    """Writes records x [n, 512] (float32 or bf16, before rotation) into a cache at rows
    dst_row [n] (int64): codes [rows, 256] uint8 + scales [rows, 512/G] uint8 (FP4), codes
    [rows, 512] uint8 + scales [rows] float32 (FP8), or codes [rows, 512] bf16 and scales None
    (BF16).  pos [n] (int64): positions whose rotary
    coordinates the records take first (None: no rotation)."""
    a = WriteArgs()
    a.n_rows = x.shape[0]
    a.x = _ptr(x)
    a.x_f32 = 1 if x.dtype == torch.float32 else 0
    if a.x_f32 == 0 and x.dtype != torch.bfloat16:
        raise ValueError("x must be float32 or bfloat16")
    a.pos = _ptr(pos)
    a.rope_theta = float(theta)
    a.dst_row = _ptr(dst_row)
    a.cache_rows = codes.shape[0]
    a.out_dtype = int(out_dtype)
    a.codes, a.scales, a.dev_status = _ptr(codes), _ptr(scales), _ptr(dev_status)
    _check(_write_records(C.byref(a), _stream()), "csa2_write_records")


def compress(kv, gate, ratio: int):
    """Entries [T // ratio, 512] float32 pooled from tokens kv, gate [T, 512] (float32 or bf16)
    with channel-wise softmax gates."""
    if kv.shape != gate.shape or kv.dtype != gate.dtype:
        raise ValueError("kv and gate must have the same shape and dtype")
    n = kv.shape[0] // ratio
    out = torch.empty((n, kv.shape[1]), dtype=torch.float32, device=kv.device)
    a = CompressArgs()
    a.n_entries, a.ratio = n, int(ratio)
    a.kv, a.gate, a.out = _ptr(kv), _ptr(gate), _ptr(out)
    a.x_f32 = 1 if kv.dtype == torch.float32 else 0
    _check(_compress(C.byref(a), _stream()), "csa2_compress")
    return out


class DecodeLayer:
    """One prepared csa2_fused_decode call: argument struct, outputs and workspace are built
    once, so that repeated calls (and CUDA-graph capture) only launch kernels."""

    def __init__(self, mode, *, q_idx=None, w=None, k_idx=None, k_scale=None, seq_of_row, n_visible, q, q_pos,
                 latents, lat_scale, swa, swa_scale, swa_pos0, window, sink, K=512, theta=1e4,
                 softmax_scale=HEAD_DIM ** -0.5, block_size=64, n_keep=64, pool=None, n_pool=None, idx=None,
                 out_dtype=torch.float32):
        self.mode = MODES[mode] if isinstance(mode, str) else int(mode)
        dev = _dev(q)
        n_rows = q.shape[0]
        self.out = torch.empty((n_rows, HEADS, HEAD_DIM), dtype=out_dtype, device=dev)
        self.sink_mass = torch.empty((n_rows, HEADS), dtype=torch.float32, device=dev)
        if self.mode == MODE_REUSE:
            if idx is None:
                raise ValueError("REUSE needs the preceding layer's idx")
            self.idx = idx
        else:
            self.idx = torch.empty((n_rows, K), dtype=torch.int32, device=dev)
        if self.mode == MODE_FULL_POOL:
            self.pool = torch.empty((n_rows, n_keep * block_size), dtype=torch.int32, device=dev)
            self.n_pool = torch.empty((n_rows,), dtype=torch.int32, device=dev)
        else:
            self.pool, self.n_pool = pool, n_pool
        a = DecodeArgs()
        a.mode, a.K, a.block_size, a.n_keep = self.mode, K, block_size, n_keep
        if self.mode != MODE_REUSE:
            a.index = _index_args(q_idx, w, k_idx, k_scale, seq_of_row, n_visible)
        a.pool, a.n_pool = _ptr(self.pool), _ptr(self.n_pool)
        a.pool_len = self.pool.shape[1] if self.pool is not None else 0
        a.idx = _ptr(self.idx)
        a.attn = _attn_args(q, q_pos, seq_of_row, latents, lat_scale, self.idx, K, swa, swa_scale, swa_pos0,
                            window, sink, theta, softmax_scale, self.out, self.sink_mass)
        nbytes = int(_decode_ws(C.byref(a)))
        self._ws, a.workspace_bytes = _ws(nbytes, dev)
        a.workspace = _ptr(self._ws)
        self._args = a
        self._keep = (q_idx, w, k_idx, k_scale, seq_of_row, n_visible, q, q_pos, latents, lat_scale, swa, swa_scale,
                      swa_pos0, sink, pool, n_pool)

    @property
    def launches(self) -> int:
        """Kernels one call launches."""
        return int(_decode_launches(C.byref(self._args)))

    def set_stage_events(self, events):
        """Record the given torch.cuda.Event objects (up to 4, None to skip) at the stage
        boundaries of every later call: before indexing, after the scan, after top-K merge /
        block pool, after attention."""
        self._events = list(events) + [None] * (4 - len(events))
        for i, ev in enumerate(self._events[:4]):
            if ev is not None and ev.cuda_event == 0:
                ev.record()  # torch creates the CUDA event lazily
            self._args.stage_events[i] = ev.cuda_event if ev is not None else None

    def __call__(self):
        _check(_fused_decode(C.byref(self._args), _stream()), "csa2_fused_decode")
        return self.out


def fused_decode(mode, **kw):
    """One CSA2 decode layer; returns the DecodeLayer after running it (outputs: .out, .sink_mass,
    .idx, .pool, .n_pool)."""
    layer = DecodeLayer(mode, **kw)
    layer()
    return layer


# ------------------------------------------------------------------ projections
def _bf16_2d(t, name):
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 tensor")
    return t


class QueryProj:
    """A prepared csa2_query_proj call (weights, output and workspace bound once):
    q [T, heads, 512] bf16 from hidden states x [T, hidden] bf16 through the low-rank path
    W_DQ [q_rank, hidden] -> RMSNorm * g_q -> W_UQ [heads * 512, q_rank] -> per-head RMSNorm
    * g_head."""

    def __init__(self, x, w_dq, w_uq, g_q=None, g_head=None, eps: float = 1e-6):
        for t, n in ((x, "x"), (w_dq, "w_dq"), (w_uq, "w_uq")):
            _bf16_2d(t, n)
        for g, n in ((g_q, "g_q"), (g_head, "g_head")):
            if g is not None and (g.dtype != torch.float32 or not g.is_contiguous()):
                raise ValueError(f"{n} must be a contiguous float32 tensor")
        T, hidden = x.shape
        q_rank = w_dq.shape[0]
        heads = w_uq.shape[0] // HEAD_DIM
        if w_dq.shape[1] != hidden or w_uq.shape[1] != q_rank or w_uq.shape[0] != heads * HEAD_DIM:
            raise ValueError("weight shapes do not match")
        self.q = torch.empty((T, heads, HEAD_DIM), dtype=torch.bfloat16, device=x.device)
        a = QueryProjArgs()
        a.n_tokens, a.hidden, a.q_rank, a.n_heads = T, hidden, q_rank, heads
        a.x, a.w_dq, a.w_uq, a.q = _ptr(x), _ptr(w_dq), _ptr(w_uq), _ptr(self.q)
        a.g_q, a.g_head, a.eps = _ptr(g_q), _ptr(g_head), float(eps)
        self._ws, a.workspace_bytes = _ws(int(_query_proj_ws(C.byref(a))), x.device)
        a.workspace = _ptr(self._ws)
        self._args = a
        self._keep = (x, w_dq, w_uq, g_q, g_head)

    def __call__(self):
        _check(_query_proj(C.byref(self._args), _stream()), "csa2_query_proj")
        return self.q


class OutProj:
    """A prepared csa2_out_proj call: out [T, hidden] bf16 from attention's output o
    [T, heads, 512] bf16 through the grouped low-rank projection W_OA [G, o_rank,
    heads / G * 512] (per group of consecutive heads), then W_OB [hidden, G * o_rank]."""

    def __init__(self, o, w_oa, w_ob):
        for t, n in ((o, "o"), (w_oa, "w_oa"), (w_ob, "w_ob")):
            _bf16_2d(t, n)
        T, heads, _ = o.shape
        G, o_rank, kg = w_oa.shape
        hidden = w_ob.shape[0]
        if kg * G != heads * HEAD_DIM or w_ob.shape[1] != G * o_rank:
            raise ValueError("weight shapes do not match")
        self.out = torch.empty((T, hidden), dtype=torch.bfloat16, device=o.device)
        a = OutProjArgs()
        a.n_tokens, a.n_heads, a.n_groups, a.o_rank, a.hidden = T, heads, G, o_rank, hidden
        a.o, a.w_oa, a.w_ob, a.out = _ptr(o), _ptr(w_oa), _ptr(w_ob), _ptr(self.out)
        self._ws, a.workspace_bytes = _ws(int(_out_proj_ws(C.byref(a))), o.device)
        a.workspace = _ptr(self._ws)
        self._args = a
        self._keep = (o, w_oa, w_ob)

    def __call__(self):
        _check(_out_proj(C.byref(self._args), _stream()), "csa2_out_proj")
        return self.out


def query_proj(x, w_dq, w_uq, g_q=None, g_head=None, eps: float = 1e-6):
    """Attention queries [T, heads, 512] bf16 of hidden states x (see QueryProj)."""
    return QueryProj(x, w_dq, w_uq, g_q, g_head, eps)()


def out_proj(o, w_oa, w_ob):
    """Hidden-size output [T, hidden] bf16 of attention's output o (see OutProj)."""
    return OutProj(o, w_oa, w_ob)()


def linear(x, w):
    """out [T, out_features] bf16 = x [T, in_features] bf16 times w [out_features,
    in_features] bf16 transposed (fp32 accumulation on the tensor cores)."""
    _bf16_2d(x, "x")
    _bf16_2d(w, "w")
    if x.shape[1] != w.shape[1]:
        raise ValueError("x and w disagree on in_features")
    out = torch.empty((x.shape[0], w.shape[0]), dtype=torch.bfloat16, device=x.device)
    a = LinearArgs()
    a.n_tokens, a.in_features, a.out_features = x.shape[0], x.shape[1], w.shape[0]
    a.x, a.w, a.out = _ptr(x), _ptr(w), _ptr(out)
    _check(_linear(C.byref(a), _stream()), "csa2_linear")
    return out


def expand_mxfp4(codes, exps):
    """MXFP4 keys (codes [..., 64] uint8, exponents [..., 4] uint8) -> their exact bf16 values
    [..., 128] (for the prefill indexer, which reuses a chunk's keys for every query)."""
    if codes.dtype != torch.uint8 or exps.dtype != torch.uint8 or codes.shape[-1] != 64 or exps.shape[-1] != 4:
        raise ValueError("expected uint8 codes [..., 64] and exponents [..., 4]")
    out = torch.empty(codes.shape[:-1] + (128,), dtype=torch.bfloat16, device=codes.device)
    a = ExpandArgs()
    a.n_records = codes.numel() // 64
    a.codes, a.exps, a.out = _ptr(codes), _ptr(exps), _ptr(out)
    _check(_expand(C.byref(a), _stream()), "csa2_expand_mxfp4")
    return out
