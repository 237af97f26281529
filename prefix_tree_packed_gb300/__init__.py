"""Python binding of the packed prefix-tree attention library (``libtreeattn.so``).

Argument marshalling only: every step of the path (planning, RoPE, attention,
readout) runs inside the C-ABI library, declared in ``include/tree_attn.h``.
Tensors are passed as raw device pointers (any object with ``data_ptr()``, or
an int) and streams as raw ``cudaStream_t`` handles; PyTorch is used by callers
for device memory and streams only.

Importing this package raises if the compiled library is missing: there is no
other implementation to fall back to.  Build it with
``python prefix_tree_packed_gb300/build.py``.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtreeattn.so")

TREE_OK = 0
TREE_ERR_INVALID_ARG = 1
TREE_ERR_BAD_TREE = 2
TREE_ERR_DEPTH = 3
TREE_ERR_ROW_TOO_LONG = 4
TREE_ERR_UNSUPPORTED = 5
TREE_ERR_CUDA = 6
TREE_ERR_TIMEOUT = 7

# every symbol the header declares
EXPORTS = (
    "tree_last_error", "tree_version", "tree_pack_plan", "tree_plan_free", "tree_plan_query",
    "tree_plan_chunk", "tree_plan_tables", "tree_plan_upload", "tree_plan_upload_staged", "tree_rope_table",
    "tree_rope",
    "tree_attn_fwd", "tree_attn_fwd_noalloc", "readout_decide", "tree_runtime_create", "tree_runtime_destroy",
    "tree_runtime_step", "tree_runtime_attach_io", "tree_runtime_step_host", "tree_shard_rows", "tree_shard_select",
    # include/tree_queue.h
    "tree_queue_default_opts", "tree_queue_create", "tree_queue_destroy", "tree_queue_push", "tree_queue_cancel",
    "tree_queue_info", "tree_queue_pop", "tree_batch_view", "tree_batch_free",
    # include/tree_layer.h
    "tree_gemm", "tree_gemm_ex", "tree_gemm_qkv", "tree_rmsnorm", "tree_layer_workspace_bytes", "tree_layer_fwd", "tree_last_layer_workspace_bytes",
    "tree_last_layer_fwd", "tree_model_workspace_bytes", "tree_model_fwd", "tree_session_create", "tree_session_run",
    "tree_session_destroy",
)

GEMM_STORE = 0
GEMM_RESIDUAL = 1
GEMM_SWIGLU = 2
GEMM_STORE_F32 = 3


class TreeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python prefix_tree_packed_gb300/build.py`")
_lib = C.CDLL(LIB_PATH)

_i32p = C.POINTER(C.c_int32)


class _Spec(C.Structure):
    _fields_ = [("n_blocks", C.c_int32), ("parent", _i32p), ("length", _i32p),
                ("key", C.POINTER(C.c_uint64)), ("resident", C.POINTER(C.c_uint8)),
                ("n_questions", C.c_int32), ("leaf1", _i32p), ("leaf2", _i32p)]


class _Block(C.Structure):
    _fields_ = [("key", C.c_uint64), ("length", C.c_int32)]


class _Request(C.Structure):
    _fields_ = [("id", C.c_int64), ("arrival_ms", C.c_double), ("n_prompts", C.c_int32),
                ("prompt_blocks", _i32p), ("blocks", C.POINTER(_Block)), ("n_questions", C.c_int32),
                ("q_prompt1", _i32p), ("q_prompt2", _i32p)]


class QueueOpts(C.Structure):
    _fields_ = [("max_batch_tokens", C.c_int32), ("long_tokens", C.c_int32), ("fifo", C.c_int32),
                ("ms_per_token", C.c_double), ("max_depth", C.c_int32), ("max_row", C.c_int32),
                ("n_resident", C.c_int32), ("resident_keys", C.POINTER(C.c_uint64))]


class _QueueInfo(C.Structure):
    _fields_ = [("n_short", C.c_int32), ("n_long", C.c_int32)]


class _BatchView(C.Structure):
    _fields_ = [("lane", C.c_int32), ("n_requests", C.c_int32), ("request_ids", C.POINTER(C.c_int64)),
                ("request_q0", _i32p), ("cost", C.c_int64), ("spec", _Spec)]


class LayerWeights(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("hq", C.c_int32), ("hkv", C.c_int32), ("d", C.c_int32), ("ffn", C.c_int32),
                ("eps", C.c_float), ("w_in", C.c_void_p), ("wqkv", C.c_void_p),
                ("wo", C.c_void_p), ("w_post", C.c_void_p), ("wgu", C.c_void_p), ("wd", C.c_void_p)]


class _Opts(C.Structure):
    _fields_ = [("max_fwd", C.c_int32), ("max_depth", C.c_int32), ("max_row", C.c_int32), ("tiling", C.c_int32),
                ("pack_heads", C.c_int32)]


class PlanInfo(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "n_input_blocks", "n_blocks", "n_tot", "n_res", "n_fwd", "n_chunks", "n_qtiles",
        "n_entries", "n_slots", "n_questions", "max_fwd", "bm", "bn", "max_pos")] + [
        ("pairs", C.c_int64), ("dev_bytes", C.c_size_t)] + [(n, C.c_size_t) for n in (
        "off_pos", "off_send", "off_qtile", "off_ent", "off_order", "off_chunk", "off_slot_tok",
        "off_r1", "off_r2", "off_runs")] + [("tiling", C.c_int32), ("off_vkeys", C.c_size_t),
                                            ("off_vruns", C.c_size_t), ("pack_heads", C.c_int32)]


class ChunkInfo(C.Structure):
    _fields_ = [("q0", C.c_int32), ("q1", C.c_int32), ("t0", C.c_int32), ("t1", C.c_int32),
                ("pairs", C.c_int64), ("n_entries", C.c_int32)]


_VIEW_FIELDS = ("block_map", "blk_start", "blk_len", "blk_parent", "blk_depth", "blk_pos0",
                "blk_send", "blk_resident", "blk_slot", "pos", "send", "chunk_q0", "chunk_q1",
                "chunk_t0", "chunk_t1", "qt_row0", "qt_row1", "qt_ent0", "qt_ent1", "ent",
                "qt_order", "slot_tok", "r1", "r2")


class _View(C.Structure):
    _fields_ = [(n, _i32p) for n in _VIEW_FIELDS] + [("image", C.c_void_p), ("image_bytes", C.c_size_t),
                                                     ("runs", _i32p), ("vkeys", _i32p), ("vruns", _i32p)]


class _Shard(C.Structure):
    _fields_ = [("n_blocks", C.c_int32), ("parent", C.c_void_p), ("length", C.c_void_p), ("key", C.c_void_p),
                ("resident", C.c_void_p), ("block_index", C.c_void_p), ("n_questions", C.c_int32),
                ("leaf1", C.c_void_p), ("leaf2", C.c_void_p), ("question_index", C.c_void_p)]


class AttnParams(C.Structure):
    _fields_ = [("hq", C.c_int32), ("hkv", C.c_int32), ("d", C.c_int32), ("scale", C.c_float),
                ("work", C.c_void_p), ("self_test", C.c_int32)]


class _StepArgs(C.Structure):
    _fields_ = [("spec", C.c_void_p), ("opts", C.c_void_p), ("q", C.c_void_p), ("k", C.c_void_p),
                ("v", C.c_void_p), ("o", C.c_void_p), ("lse", C.c_void_p), ("cos_sin", C.c_void_p),
                ("max_pos", C.c_int32), ("hq", C.c_int32), ("hkv", C.c_int32), ("d", C.c_int32),
                ("scale", C.c_float), ("logits", C.c_void_p), ("stride", C.c_int32), ("n_letters", C.c_void_p),
                ("temperature", C.c_void_p), ("p_cal", C.c_void_p), ("p_avg", C.c_void_p), ("choice", C.c_void_p),
                ("status", C.c_void_p), ("attn_events", C.c_void_p * 2)]


class IoCaps(C.Structure):
    """``tree_io_caps_t``: sizes of the runtime's device sets for host-buffer steps."""
    _fields_ = [(n, C.c_int32) for n in ("max_fwd", "max_tot", "hq", "hkv", "d", "stride", "max_slots",
                                         "max_questions")]


class _HostStepArgs(C.Structure):
    _fields_ = [("spec", C.c_void_p), ("opts", C.c_void_p), ("q", C.c_void_p), ("k", C.c_void_p),
                ("v", C.c_void_p), ("o", C.c_void_p), ("cos_sin", C.c_void_p), ("max_pos", C.c_int32),
                ("scale", C.c_float), ("logits", C.c_void_p), ("n_letters", C.c_void_p),
                ("temperature", C.c_void_p), ("p_cal", C.c_void_p), ("p_avg", C.c_void_p), ("choice", C.c_void_p),
                ("status", C.c_void_p)]


_vp = C.c_void_p
_lib.tree_last_error.restype = C.c_char_p
_lib.tree_version.restype = C.c_int
_lib.tree_pack_plan.argtypes = [C.POINTER(_Spec), C.POINTER(_Opts), C.POINTER(_vp)]
_lib.tree_plan_free.argtypes = [_vp]
_lib.tree_plan_query.argtypes = [_vp, C.POINTER(PlanInfo)]
_lib.tree_plan_chunk.argtypes = [_vp, C.c_int32, C.POINTER(ChunkInfo)]
_lib.tree_plan_tables.argtypes = [_vp, C.POINTER(_View)]
_lib.tree_plan_upload.argtypes = [_vp, _vp, C.c_size_t, _vp]
_lib.tree_plan_upload_staged.argtypes = [_vp, _vp, C.c_size_t, _vp, C.c_size_t, _vp]
_lib.tree_rope_table.argtypes = [_vp, C.c_int32, C.c_int32, C.c_double]
_lib.tree_rope.argtypes = [_vp, _vp, C.c_int32, _vp, _vp, C.c_int32, C.c_int32, C.c_int32, _vp,
                           C.c_int32, _vp, _vp]
_lib.tree_attn_fwd.argtypes = [_vp, _vp, C.c_int32, _vp, _vp, _vp, _vp, _vp, C.POINTER(AttnParams),
                               _vp, _vp]
_lib.tree_attn_fwd_noalloc.argtypes = [_vp, _vp, C.c_int32, _vp, _vp, _vp, _vp, _vp, C.POINTER(AttnParams),
                                       _vp, _vp]
_lib.tree_shard_rows.argtypes = [C.POINTER(_Spec), C.POINTER(_Opts), C.c_int32, _vp, _vp, _vp]
_lib.tree_shard_select.argtypes = [C.POINTER(_Spec), _vp, _vp, C.c_int32, C.POINTER(_Shard)]
_lib.readout_decide.argtypes = [_vp, C.c_int32, _vp, _vp, _vp, _vp, C.c_int32, _vp, _vp, _vp, _vp, _vp]
_lib.tree_runtime_create.argtypes = [C.c_size_t, C.c_int32, C.POINTER(_vp)]
_lib.tree_runtime_destroy.argtypes = [_vp]
_lib.tree_runtime_step.argtypes = [_vp, C.POINTER(_StepArgs), C.POINTER(PlanInfo), _vp]
_lib.tree_runtime_attach_io.argtypes = [_vp, C.POINTER(IoCaps)]
_lib.tree_runtime_step_host.argtypes = [_vp, C.POINTER(_HostStepArgs), C.POINTER(PlanInfo), _vp]
_lib.tree_gemm.argtypes = [_vp, _vp, _vp, _vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _vp, _vp]
_lib.tree_gemm_ex.argtypes = [_vp, _vp, _vp, _vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _vp, _vp]
_lib.tree_gemm_qkv.argtypes = [_vp, _vp, _vp, _vp, _vp, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _vp, _vp]
_lib.tree_rmsnorm.argtypes = [_vp, _vp, _vp, C.c_int32, C.c_int32, C.c_float, _vp]
_lib.tree_layer_workspace_bytes.argtypes = [_vp, C.POINTER(LayerWeights), C.POINTER(C.c_size_t)]
_lib.tree_layer_fwd.argtypes = [_vp, _vp, C.POINTER(LayerWeights), _vp, _vp, _vp, _vp, _vp, C.c_int32, _vp, C.c_size_t,
                                _vp, _vp, _vp]
_lib.tree_last_layer_workspace_bytes.argtypes = [_vp, C.POINTER(LayerWeights), C.POINTER(C.c_size_t)]
_lib.tree_last_layer_fwd.argtypes = [_vp, _vp, C.POINTER(LayerWeights), _vp, _vp, _vp, _vp, C.c_int32, _vp, _vp,
                                     C.c_int32, _vp, _vp, C.c_size_t, _vp, _vp, _vp]
_lib.tree_model_workspace_bytes.argtypes = [_vp, C.POINTER(LayerWeights), C.POINTER(C.c_size_t)]
_lib.tree_model_fwd.argtypes = [_vp, _vp, C.POINTER(LayerWeights), C.c_int32, _vp, C.POINTER(_vp), C.POINTER(_vp),
                                _vp, C.c_int32, _vp, _vp, C.c_int32, _vp, _vp, C.c_size_t, _vp, _vp, _vp]
_lib.tree_session_create.argtypes = [_vp, _vp, C.POINTER(LayerWeights), C.c_int32, _vp, C.POINTER(_vp),
                                     C.POINTER(_vp), _vp, C.c_int32, _vp, _vp, C.c_int32, _vp, _vp, C.c_size_t, _vp,
                                     _vp, C.POINTER(_vp)]
_lib.tree_session_run.argtypes = [_vp, C.c_double, _vp, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
_lib.tree_session_destroy.argtypes = [_vp]
_lib.tree_queue_default_opts.argtypes = [C.POINTER(QueueOpts)]
_lib.tree_queue_create.argtypes = [C.POINTER(QueueOpts), C.POINTER(_vp)]
_lib.tree_queue_destroy.argtypes = [_vp]
_lib.tree_queue_push.argtypes = [_vp, C.POINTER(_Request), C.POINTER(C.c_int64)]
_lib.tree_queue_cancel.argtypes = [_vp, C.c_int64]
_lib.tree_queue_info.argtypes = [_vp, C.POINTER(_QueueInfo)]
_lib.tree_queue_pop.argtypes = [_vp, C.c_double, C.POINTER(_vp)]
_lib.tree_batch_view.argtypes = [_vp, C.POINTER(_BatchView)]
_lib.tree_batch_free.argtypes = [_vp]
for _f in ("tree_gemm", "tree_gemm_ex", "tree_gemm_qkv", "tree_rmsnorm", "tree_layer_workspace_bytes", "tree_layer_fwd",
           "tree_last_layer_workspace_bytes", "tree_last_layer_fwd", "tree_model_workspace_bytes", "tree_model_fwd",
           "tree_session_create", "tree_session_run", "tree_session_destroy",
           "tree_runtime_create", "tree_runtime_destroy", "tree_runtime_step", "tree_runtime_attach_io",
           "tree_runtime_step_host", "tree_queue_default_opts",
           "tree_queue_create", "tree_queue_destroy", "tree_queue_push", "tree_queue_cancel", "tree_queue_info",
           "tree_queue_pop", "tree_batch_view", "tree_batch_free"):
    getattr(_lib, _f).restype = C.c_int
for _f in ("tree_pack_plan", "tree_plan_free", "tree_plan_query", "tree_plan_chunk", "tree_plan_tables",
           "tree_plan_upload", "tree_plan_upload_staged", "tree_rope_table", "tree_rope", "tree_attn_fwd", "tree_attn_fwd_noalloc",
           "readout_decide", "tree_shard_rows", "tree_shard_select"):
    getattr(_lib, _f).restype = C.c_int


def _check(rc: int):
    if rc != TREE_OK:
        raise TreeError(rc, _lib.tree_last_error().decode(errors="replace"))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def version() -> int:
    return _lib.tree_version()


class Spec:
    """A batch's forest as the planner reads it (arrays kept alive, struct built once)."""

    def __init__(self, parent, length, key=None, resident=None, leaf1=None, leaf2=None,
                 max_fwd: int = 0, max_depth: int = 0, max_row: int = 0, tiling: int = 0, pack_heads: int = 0):
        self._keep = []
        par = np.ascontiguousarray(parent, np.int32)
        ln = np.ascontiguousarray(length, np.int32)
        self.spec = _Spec()
        self.spec.n_blocks = par.shape[0]
        self.spec.parent = par.ctypes.data_as(_i32p)
        self.spec.length = ln.ctypes.data_as(_i32p)
        self._keep += [par, ln]
        if key is not None:
            k = np.ascontiguousarray(key, np.uint64)
            self.spec.key = k.ctypes.data_as(C.POINTER(C.c_uint64))
            self._keep.append(k)
        if resident is not None:
            r = np.ascontiguousarray(resident, np.uint8)
            self.spec.resident = r.ctypes.data_as(C.POINTER(C.c_uint8))
            self._keep.append(r)
        if leaf1 is not None:
            l1 = np.ascontiguousarray(leaf1, np.int32)
            l2 = np.ascontiguousarray(leaf2, np.int32)
            self.spec.n_questions = l1.shape[0]
            self.spec.leaf1 = l1.ctypes.data_as(_i32p)
            self.spec.leaf2 = l2.ctypes.data_as(_i32p)
            self._keep += [l1, l2]
        self.opts = _Opts(max_fwd, max_depth, max_row, tiling, pack_heads)

    @classmethod
    def from_forest(cls, forest, **kw):
        return cls(forest.parent, forest.length, forest.key, forest.resident, **kw)


def shard_rows(spec: Spec, n_ranks: int):
    """tree_shard_rows: (block_rank [n_blocks], question_rank [n_questions], rank_pairs [n_ranks])."""
    nb, nq = spec.spec.n_blocks, spec.spec.n_questions
    block_rank = np.empty(nb, np.int32)
    question_rank = np.empty(max(nq, 1), np.int32)
    pairs = np.empty(n_ranks, np.int64)
    _check(_lib.tree_shard_rows(C.byref(spec.spec), C.byref(spec.opts), n_ranks, block_rank.ctypes.data,
                                question_rank.ctypes.data, pairs.ctypes.data))
    return block_rank, question_rank[:nq], pairs


def shard_select(spec: Spec, block_rank, question_rank, rank: int) -> dict:
    """tree_shard_select: the rank's blocks and questions as arrays (parent, length, key, resident,
    block_index, leaf1, leaf2, question_index), in input order."""
    nb, nq = spec.spec.n_blocks, spec.spec.n_questions
    br = np.ascontiguousarray(block_rank, np.int32)
    qr = np.ascontiguousarray(question_rank, np.int32) if nq else np.zeros(1, np.int32)
    out = dict(parent=np.empty(nb, np.int32), length=np.empty(nb, np.int32), key=np.empty(nb, np.uint64),
               resident=np.empty(nb, np.uint8), block_index=np.empty(nb, np.int32),
               leaf1=np.empty(max(nq, 1), np.int32), leaf2=np.empty(max(nq, 1), np.int32),
               question_index=np.empty(max(nq, 1), np.int32))
    sh = _Shard(0, *(out[k].ctypes.data for k in ("parent", "length", "key", "resident", "block_index")), 0,
                *(out[k].ctypes.data for k in ("leaf1", "leaf2", "question_index")))
    _check(_lib.tree_shard_select(C.byref(spec.spec), br.ctypes.data, qr.ctypes.data, rank, C.byref(sh)))
    for k in ("parent", "length", "key", "resident", "block_index"):
        out[k] = out[k][:sh.n_blocks]
    for k in ("leaf1", "leaf2", "question_index"):
        out[k] = out[k][:sh.n_questions]
    return out


def gemm(a, b, c, m: int, n: int, k: int, epi: int = GEMM_STORE, r=None, status=None, stream=None, tile_n: int = 0):
    """tree_gemm_ex: C[m, n] = epilogue(A[m, k] B^T), f16 in and out, f32 accumulation (tile_n 0: automatic)."""
    _check(_lib.tree_gemm_ex(_ptr(a), _ptr(b), _ptr(c), _ptr(r), m, n, k, epi, tile_n, _ptr(status), _stream(stream)))


def gemm_qkv(a, wqkv, q, k, v, m: int, nq: int, nkv: int, kdim: int, status=None, stream=None):
    """tree_gemm_qkv: the q, k, v projections in one GEMM, written to three outputs."""
    _check(_lib.tree_gemm_qkv(_ptr(a), _ptr(wqkv), _ptr(q), _ptr(k), _ptr(v), m, nq, nkv, kdim, _ptr(status),
                              _stream(stream)))


def rmsnorm(x, w, y, rows: int, cols: int, eps: float = 1e-5, stream=None):
    """tree_rmsnorm: y = f16(f16(x / sqrt(mean(x^2) + eps)) * w) per row."""
    _check(_lib.tree_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, cols, eps, _stream(stream)))


def layer_weights(hidden: int, hq: int, hkv: int, d: int, ffn: int, tensors: dict, eps: float = 1e-5) -> LayerWeights:
    """LayerWeights from device tensors keyed w_in, wqkv, wo, w_post, wgu, wd (kept alive by the caller)."""
    return LayerWeights(hidden, hq, hkv, d, ffn, eps, *[_ptr(tensors[k]) for k in
                                                        ("w_in", "wqkv", "wo", "w_post", "wgu", "wd")])


def layer_workspace_bytes(plan: "Plan", w: LayerWeights) -> int:
    n = C.c_size_t()
    _check(_lib.tree_layer_workspace_bytes(plan.handle, C.byref(w), C.byref(n)))
    return int(n.value)


def layer_fwd(plan: "Plan", plan_dev, w: LayerWeights, x, k_cache, v_cache, y, cos_sin, max_pos: int, workspace,
              workspace_bytes: int, work=None, status=None, stream=None):
    """tree_layer_fwd: one Llama layer over the plan's forward tokens (see include/tree_layer.h)."""
    _check(_lib.tree_layer_fwd(plan.handle, _ptr(plan_dev), C.byref(w), _ptr(x), _ptr(k_cache), _ptr(v_cache), _ptr(y),
                               _ptr(cos_sin), max_pos, _ptr(workspace), workspace_bytes, _ptr(work), _ptr(status),
                               _stream(stream)))


def last_layer_workspace_bytes(plan: "Plan", w: LayerWeights) -> int:
    n = C.c_size_t()
    _check(_lib.tree_last_layer_workspace_bytes(plan.handle, C.byref(w), C.byref(n)))
    return int(n.value)


def last_layer_fwd(plan: "Plan", plan_dev, w: LayerWeights, x, k_cache, v_cache, cos_sin, max_pos: int, w_final,
                   w_letters, stride: int, logits, workspace, workspace_bytes: int, work=None, status=None,
                   stream=None):
    """tree_last_layer_fwd: the final layer, pruned to the readout rows, and the letter logits (f32)."""
    _check(_lib.tree_last_layer_fwd(plan.handle, _ptr(plan_dev), C.byref(w), _ptr(x), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(cos_sin), max_pos, _ptr(w_final), _ptr(w_letters), stride, _ptr(logits),
                                    _ptr(workspace), workspace_bytes, _ptr(work), _ptr(status), _stream(stream)))


def model_workspace_bytes(plan: "Plan", w: LayerWeights) -> int:
    n = C.c_size_t()
    _check(_lib.tree_model_workspace_bytes(plan.handle, C.byref(w), C.byref(n)))
    return int(n.value)


def model_fwd(plan: "Plan", plan_dev, layers, x, k_caches, v_caches, cos_sin, max_pos: int, w_final, w_letters,
              stride: int, logits, workspace, workspace_bytes: int, work=None, status=None, stream=None):
    """tree_model_fwd: every layer (the last pruned to the readout rows) and the letter logits."""
    n = len(layers)
    arr = (LayerWeights * n)(*layers)
    kc = (_vp * n)(*[_ptr(t) for t in k_caches])
    vc = (_vp * n)(*[_ptr(t) for t in v_caches])
    _check(_lib.tree_model_fwd(plan.handle, _ptr(plan_dev), arr, n, _ptr(x), kc, vc, _ptr(cos_sin), max_pos,
                               _ptr(w_final), _ptr(w_letters), stride, _ptr(logits), _ptr(workspace), workspace_bytes,
                               _ptr(work), _ptr(status), _stream(stream)))


class Session:
    """``tree_session``: a decision forward of the long-request lane, run in slices of whole layers."""

    def __init__(self, plan: "Plan", plan_dev, layers, x, k_caches, v_caches, cos_sin, max_pos: int, w_final,
                 w_letters, stride: int, logits, workspace, workspace_bytes: int, work=None, status=None):
        n = len(layers)
        self._arr = (LayerWeights * n)(*layers)
        kc = (_vp * n)(*[_ptr(t) for t in k_caches])
        vc = (_vp * n)(*[_ptr(t) for t in v_caches])
        self._s = _vp()
        _check(_lib.tree_session_create(plan.handle, _ptr(plan_dev), self._arr, n, _ptr(x), kc, vc, _ptr(cos_sin),
                                        max_pos, _ptr(w_final), _ptr(w_letters), stride, _ptr(logits),
                                        _ptr(workspace), workspace_bytes, _ptr(work), _ptr(status), C.byref(self._s)))

    def run(self, slice_ms: float, stream=None) -> tuple[int, bool]:
        """Run whole layers until slice_ms of wall time has passed; returns (layers run, done)."""
        ran, done = C.c_int32(), C.c_int32()
        _check(_lib.tree_session_run(self._s, float(slice_ms), _stream(stream), C.byref(ran), C.byref(done)))
        return int(ran.value), bool(done.value)

    def close(self):
        if self._s:
            _lib.tree_session_destroy(self._s)
            self._s = _vp()

    def __del__(self):
        self.close()


def queue_default_opts() -> QueueOpts:
    o = QueueOpts()
    _check(_lib.tree_queue_default_opts(C.byref(o)))
    return o


class Batch:
    """One batch taken from a ``Queue``: its requests and its forest (``spec``), copied out."""

    def __init__(self, view: _BatchView):
        n = view.n_requests
        nb = view.spec.n_blocks
        nq = view.spec.n_questions
        self.lane = int(view.lane)
        self.cost = int(view.cost)
        self.request_ids = [int(view.request_ids[i]) for i in range(n)]
        self.request_q0 = np.array([view.request_q0[i] for i in range(n + 1)], np.int32)
        self.parent = np.array([view.spec.parent[i] for i in range(nb)], np.int32)
        self.length = np.array([view.spec.length[i] for i in range(nb)], np.int32)
        self.key = np.array([view.spec.key[i] for i in range(nb)], np.uint64)
        self.resident = np.array([view.spec.resident[i] for i in range(nb)], np.uint8)
        self.leaf1 = np.array([view.spec.leaf1[i] for i in range(nq)], np.int32)
        self.leaf2 = np.array([view.spec.leaf2[i] for i in range(nq)], np.int32)

    def spec(self, **kw) -> "Spec":
        return Spec(self.parent, self.length, self.key, self.resident, self.leaf1, self.leaf2, **kw)


class Queue:
    """``tree_queue``: HRRN / FIFO request queue with a long-request lane, batches as prefix-tree forests."""

    def __init__(self, opts: QueueOpts | None = None, resident_keys=()):
        o = queue_default_opts() if opts is None else opts
        keys = np.ascontiguousarray(list(resident_keys), np.uint64)
        o.n_resident = keys.shape[0]
        o.resident_keys = keys.ctypes.data_as(C.POINTER(C.c_uint64)) if keys.shape[0] else None
        self._q = _vp()
        _check(_lib.tree_queue_create(C.byref(o), C.byref(self._q)))

    def close(self):
        if self._q:
            _lib.tree_queue_destroy(self._q)
            self._q = _vp()

    def __del__(self):
        self.close()

    def push(self, rid: int, arrival_ms: float, prompts, questions=()) -> int:
        """prompts: list of [(key, length), ...] root first; questions: [(prompt1, prompt2), ...]. Returns the cost."""
        counts = np.array([len(p) for p in prompts], np.int32)
        blocks = (_Block * max(int(counts.sum()), 1))()
        i = 0
        for p in prompts:
            for key, length in p:
                blocks[i].key = int(key)
                blocks[i].length = int(length)
                i += 1
        q1 = np.array([a for a, _ in questions], np.int32)
        q2 = np.array([b for _, b in questions], np.int32)
        r = _Request(int(rid), float(arrival_ms), counts.shape[0], counts.ctypes.data_as(_i32p), blocks,
                     q1.shape[0], q1.ctypes.data_as(_i32p), q2.ctypes.data_as(_i32p))
        cost = C.c_int64()
        _check(_lib.tree_queue_push(self._q, C.byref(r), C.byref(cost)))
        return int(cost.value)

    def cancel(self, rid: int):
        _check(_lib.tree_queue_cancel(self._q, int(rid)))

    def info(self) -> tuple[int, int]:
        i = _QueueInfo()
        _check(_lib.tree_queue_info(self._q, C.byref(i)))
        return int(i.n_short), int(i.n_long)

    def pop(self, now_ms: float) -> Batch | None:
        b = _vp()
        _check(_lib.tree_queue_pop(self._q, float(now_ms), C.byref(b)))
        if not b:
            return None
        try:
            v = _BatchView()
            _check(_lib.tree_batch_view(b, C.byref(v)))
            return Batch(v)
        finally:
            _lib.tree_batch_free(b)


class Runtime:
    """``tree_runtime``: the whole path of one batch per ``step`` call, on one stream."""

    def __init__(self, max_plan_bytes: int, max_chunks: int):
        h = _vp()
        _check(_lib.tree_runtime_create(max_plan_bytes, max_chunks, C.byref(h)))
        self.handle = h
        self.info = PlanInfo()

    def close(self):
        h = getattr(self, "handle", None)
        if h:
            _lib.tree_runtime_destroy(h)
            self.handle = None

    __del__ = close

    def step(self, spec: Spec, q, k, v, o, cos_sin, max_pos: int, hq: int, hkv: int, d: int, logits=None,
             stride: int = 0, n_letters=None, temperature=None, p_cal=None, p_avg=None, choice=None,
             lse=None, status=None, stream=None, scale: float = 0.0, attn_events=None) -> PlanInfo:
        """attn_events: optional pair of torch.cuda.Event recorded around the step's attention launches."""
        a = _StepArgs(C.addressof(spec.spec), C.addressof(spec.opts), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                      _ptr(cos_sin), max_pos, hq, hkv, d, scale, _ptr(logits), stride, _ptr(n_letters),
                      _ptr(temperature), _ptr(p_cal), _ptr(p_avg), _ptr(choice), _ptr(status))
        if attn_events is not None:
            h0, h1 = attn_events[0].cuda_event, attn_events[1].cuda_event
            if not h0 or not h1:
                raise ValueError("attn_events: record each event once first (torch creates them lazily)")
            a.attn_events[0], a.attn_events[1] = h0, h1
        _check(_lib.tree_runtime_step(self.handle, C.byref(a), C.byref(self.info), _stream(stream)))
        return self.info

    def attach_io(self, max_fwd: int, max_tot: int, hq: int, hkv: int, d: int, stride: int = 0,
                  max_slots: int = 0, max_questions: int = 0):
        """Two device input/output sets and a copy stream for ``step_host`` (synchronises the device)."""
        self.caps = IoCaps(max_fwd, max_tot, hq, hkv, d, stride, max_slots, max_questions)
        _check(_lib.tree_runtime_attach_io(self.handle, C.byref(self.caps)))

    def step_host(self, spec: Spec, q, k, v, cos_sin, max_pos: int, o=None, logits=None, n_letters=None,
                  temperature=None, p_cal=None, p_avg=None, choice=None, status=None, stream=None,
                  scale: float = 0.0) -> PlanInfo:
        """One batch whose inputs and outputs are host buffers (page-locked torch tensors or raw
        addresses).  Returns once enqueued: the outputs are valid after ``stream`` completes."""
        a = _HostStepArgs(C.addressof(spec.spec), C.addressof(spec.opts), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                          _ptr(cos_sin), max_pos, scale, _ptr(logits), _ptr(n_letters), _ptr(temperature),
                          _ptr(p_cal), _ptr(p_avg), _ptr(choice), _ptr(status))
        _check(_lib.tree_runtime_step_host(self.handle, C.byref(a), C.byref(self.info), _stream(stream)))
        return self.info


class Plan:
    """A packed batch: owns the library's host plan (``tree_pack_plan``)."""

    def __init__(self, parent, length, key=None, resident=None, leaf1=None, leaf2=None,
                 max_fwd: int = 0, max_depth: int = 0, max_row: int = 0, tiling: int = 0, pack_heads: int = 0):
        self._keep = []
        par = np.ascontiguousarray(parent, np.int32)
        ln = np.ascontiguousarray(length, np.int32)
        spec = _Spec()
        spec.n_blocks = par.shape[0]
        spec.parent = par.ctypes.data_as(_i32p)
        spec.length = ln.ctypes.data_as(_i32p)
        self._keep += [par, ln]
        if key is not None:
            k = np.ascontiguousarray(key, np.uint64)
            spec.key = k.ctypes.data_as(C.POINTER(C.c_uint64))
            self._keep.append(k)
        if resident is not None:
            r = np.ascontiguousarray(resident, np.uint8)
            spec.resident = r.ctypes.data_as(C.POINTER(C.c_uint8))
            self._keep.append(r)
        if leaf1 is not None:
            l1 = np.ascontiguousarray(leaf1, np.int32)
            l2 = np.ascontiguousarray(leaf2, np.int32)
            spec.n_questions = l1.shape[0]
            spec.leaf1 = l1.ctypes.data_as(_i32p)
            spec.leaf2 = l2.ctypes.data_as(_i32p)
            self._keep += [l1, l2]
        opts = _Opts(max_fwd, max_depth, max_row, tiling, pack_heads)
        h = _vp()
        _check(_lib.tree_pack_plan(C.byref(spec), C.byref(opts), C.byref(h)))
        self._keep = []
        self.handle = h
        self.info = PlanInfo()
        _check(_lib.tree_plan_query(self.handle, C.byref(self.info)))

    @classmethod
    def from_forest(cls, forest, **kw):
        return cls(forest.parent, forest.length, forest.key, forest.resident, **kw)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            _lib.tree_plan_free(h)
            self.handle = None

    def chunk(self, c: int) -> ChunkInfo:
        ci = ChunkInfo()
        _check(_lib.tree_plan_chunk(self.handle, c, C.byref(ci)))
        return ci

    def tables(self) -> dict:
        """Copies of every host table as numpy arrays (plus the device image bytes)."""
        v = _View()
        _check(_lib.tree_plan_tables(self.handle, C.byref(v)))
        i = self.info
        n_kvt = -(-i.n_tot // i.bn)
        sizes = dict(block_map=i.n_input_blocks, pos=i.n_tot, send=n_kvt * i.bn, ent=i.n_entries,
                     qt_order=i.n_qtiles, slot_tok=i.n_slots, r1=i.n_questions, r2=i.n_questions)
        for n in ("blk_start", "blk_len", "blk_parent", "blk_depth", "blk_pos0", "blk_send",
                  "blk_resident", "blk_slot"):
            sizes[n] = i.n_blocks
        for n in ("chunk_q0", "chunk_q1", "chunk_t0", "chunk_t1"):
            sizes[n] = i.n_chunks
        for n in ("qt_row0", "qt_row1", "qt_ent0", "qt_ent1"):
            sizes[n] = i.n_qtiles
        out = {}
        for n in _VIEW_FIELDS:
            cnt = sizes[n]
            p = getattr(v, n)
            out[n] = np.ctypeslib.as_array(p, shape=(cnt,)).copy() if cnt > 0 else np.zeros(0, np.int32)
        out["image"] = np.ctypeslib.as_array(C.cast(v.image, C.POINTER(C.c_uint8)),
                                             shape=(v.image_bytes,)).copy()
        out["runs"] = np.ctypeslib.as_array(v.runs, shape=(n_kvt, 84)).copy()
        if i.tiling != 0 and i.n_entries > 0:
            out["vkeys"] = np.ctypeslib.as_array(v.vkeys, shape=(i.n_entries, 128)).copy()
            out["vruns"] = np.ctypeslib.as_array(v.vruns, shape=(i.n_entries, 72)).copy()
        return out

    def upload(self, dev_buf, nbytes: int, stream=None):
        _check(_lib.tree_plan_upload(self.handle, _ptr(dev_buf), nbytes, _stream(stream)))

    def upload_staged(self, dev_buf, nbytes: int, host_staging, staging_bytes: int, stream=None):
        """Upload through caller-owned page-locked host memory (never waits for the GPU)."""
        _check(_lib.tree_plan_upload_staged(self.handle, _ptr(dev_buf), nbytes, _ptr(host_staging),
                                            staging_bytes, _stream(stream)))


def rope_table(max_pos: int, d: int, theta: float) -> np.ndarray:
    out = np.empty((max_pos, d // 2, 2), np.float32)
    _check(_lib.tree_rope_table(out.ctypes.data, max_pos, d, theta))
    return out


def tree_rope(plan: Plan, plan_dev, chunk: int, q, k, hq: int, hkv: int, d: int, cos_sin,
              max_pos: int, stream=None, status=None):
    """Rotate the chunk's queries and keys in place (q=None: keys only)."""
    _check(_lib.tree_rope(plan.handle, _ptr(plan_dev), chunk, _ptr(q), _ptr(k), hq, hkv, d,
                          _ptr(cos_sin), max_pos, _ptr(status), _stream(stream)))


def tree_attn_fwd(plan: Plan, plan_dev, chunk: int, q, k, v, o, lse, hq: int, hkv: int, d: int,
                  scale: float = 0.0, status=None, stream=None, work=None, self_test: bool = False):
    """self_test=True: exercise the device-side timeout (status gets TREE_ERR_TIMEOUT, no output)."""
    p = AttnParams(hq, hkv, d, scale, _ptr(work), 1 if self_test else 0)
    _check(_lib.tree_attn_fwd(plan.handle, _ptr(plan_dev), chunk, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                              _ptr(lse), C.byref(p), _ptr(status), _stream(stream)))


def tree_attn_fwd_noalloc(plan: Plan, plan_dev, chunk: int, q, k, v, o, lse, hq: int, hkv: int, d: int,
                          scale: float = 0.0, status=None, stream=None):
    """tree_attn_fwd with the work counters kept inside the library (nothing allocated)."""
    p = AttnParams(hq, hkv, d, scale, None)
    _check(_lib.tree_attn_fwd_noalloc(plan.handle, _ptr(plan_dev), chunk, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                      _ptr(lse), C.byref(p), _ptr(status), _stream(stream)))


def readout_decide(logits, stride: int, r1, r2, n_letters, temperature, n_q: int, p_cal, p_avg=None,
                   choice=None, status=None, stream=None):
    _check(_lib.readout_decide(_ptr(logits), stride, _ptr(r1), _ptr(r2), _ptr(n_letters),
                               _ptr(temperature), n_q, _ptr(p_cal), _ptr(p_avg), _ptr(choice),
                               _ptr(status), _stream(stream)))
