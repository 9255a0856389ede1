"""ctypes binding over libpadoc.so: argument marshalling only.

Every computation runs in the library's CUDA kernels.  The names mirror the C
functions declared in include/padoc.h.  Tensors may be torch tensors (their
data_ptr() is passed) or raw integer device addresses.  There is no CPU path:
if the compiled library is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpadoc.so")

OK, ERR_INVALID, ERR_OOM, ERR_CUDA, ERR_UNSUPPORTED, ERR_DEVICE_TIMEOUT = 0, -1, -2, -3, -4, -5
F32, BF16 = 0, 1
PACK_CANONICAL, PACK_DOCUMENT = 0, 1

EXPORTED = [
    "padoc_last_error", "padoc_version", "padoc_tree_desc_build", "padoc_tree_desc_free",
    "padoc_tree_desc_info", "padoc_tree_desc_segments", "padoc_tree_desc_upload",
    "padoc_tree_attn_varlen", "padoc_kv_pool_create", "padoc_kv_pool_destroy", "padoc_kv_alloc",
    "padoc_kv_append", "padoc_kv_fork", "padoc_kv_release", "padoc_kv_seq_info", "padoc_kv_seq_blocks",
    "padoc_kv_block_refcount", "padoc_kv_pool_stats", "padoc_kv_pool_sync", "padoc_kv_pool_device",
    "padoc_debug_kv_pool_rehome", "padoc_debug_set_wait_limit", "padoc_branch_decode_ws_size", "padoc_branch_decode", "padoc_tree_mask_build", "padoc_depths",
    "padoc_device_status", "padoc_decode_plan_create", "padoc_decode_plan_ws_size", "padoc_decode_plan_fused", "padoc_decode_plan_upload",
    "padoc_decode_prefix_pass", "padoc_decode_own_pass", "padoc_decode_plan_free", "padoc_branch_decode_noalloc",
    "padoc_verify_accept", "padoc_kv_commit", "padoc_draft_index_create", "padoc_draft_index_free",
    "padoc_draft_trie", "padoc_draft_trie_batch", "padoc_tree_attn_varlen_bwd_ws_size",
    "padoc_tree_attn_varlen_bwd", "padoc_tree_desc_bwd_plan", "padoc_kv_reserve", "padoc_kv_advance", "padoc_kv_trim",
    "padoc_sched_create", "padoc_sched_destroy", "padoc_sched_submit", "padoc_sched_schedule", "padoc_sched_update",
    "padoc_sched_request", "padoc_sched_output",
]
NOALLOC_SCRATCH_BYTES = 32 << 20


class PadocError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libpadoc error {code}: {msg}")
        self.code = code


class TreeSpec(C.Structure):
    _fields_ = [("n_pages", C.c_int32), ("prefix_len", C.POINTER(C.c_int32)),
                ("n_regions", C.POINTER(C.c_int32)), ("layout_len", C.POINTER(C.c_int32)),
                ("content_len", C.POINTER(C.c_int32)), ("order", C.c_int32)]


class SchedConfig(C.Structure):
    _fields_ = [("tau", C.c_float), ("n_max", C.c_int32), ("window", C.c_int32), ("max_len", C.c_int32),
                ("fork_token", C.c_int32), ("child_token", C.c_int32), ("eos_token", C.c_int32)]


class SchedStep(C.Structure):
    _fields_ = [("cap", C.c_int32), ("n_admitted", C.c_int32), ("n_preempted", C.c_int32), ("n_active", C.c_int32),
                ("n_pages", C.c_int32), ("admitted", C.POINTER(C.c_int32)), ("preempted", C.POINTER(C.c_int32)),
                ("active", C.POINTER(C.c_int32)), ("active_seq", C.POINTER(C.c_int32)),
                ("page_seq", C.POINTER(C.c_int32)), ("branch_offsets", C.POINTER(C.c_int32))]


class DecodeBatch(C.Structure):
    _fields_ = [("n_pages", C.c_int32), ("n_branches", C.c_int32), ("page_seq", C.POINTER(C.c_int32)),
                ("branch_offsets", C.POINTER(C.c_int32)), ("branch_seq", C.POINTER(C.c_int32)),
                ("q_offsets", C.POINTER(C.c_int32))]


_lib = None


def lib() -> C.CDLL:
    """Loads libpadoc.so (built by tree_structured_shared_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run tree_structured_shared_gb300.build first")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
        p32, p64 = C.POINTER(C.c_int32), C.POINTER(C.c_int64)
        sig = {
            "padoc_last_error": (C.c_char_p, []),
            "padoc_version": (C.c_int, []),
            "padoc_tree_desc_build": (C.c_int, [C.POINTER(TreeSpec), C.POINTER(vp)]),
            "padoc_tree_desc_free": (C.c_int, [vp]),
            "padoc_tree_desc_info": (C.c_int, [vp, p64, p64, p64, p64]),
            "padoc_tree_desc_segments": (C.c_int, [vp, p32, p32]),
            "padoc_tree_desc_upload": (C.c_int, [vp, i32]),
            "padoc_tree_attn_varlen": (C.c_int, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, vp]),
            "padoc_kv_pool_create": (C.c_int, [C.POINTER(vp), vp, vp, i32, i32, i32, i32, i32, i32, i32]),
            "padoc_kv_pool_destroy": (C.c_int, [vp]),
            "padoc_kv_alloc": (C.c_int, [vp, i32, p32]),
            "padoc_kv_append": (C.c_int, [vp, i32, vp, vp, i32, vp]),
            "padoc_kv_fork": (C.c_int, [vp, i32, i32, p32]),
            "padoc_kv_release": (C.c_int, [vp, i32]),
            "padoc_kv_seq_info": (C.c_int, [vp, i32, p32, p32, p32]),
            "padoc_kv_seq_blocks": (C.c_int, [vp, i32, p32, i32]),
            "padoc_kv_block_refcount": (C.c_int, [vp, i32, p32]),
            "padoc_kv_pool_stats": (C.c_int, [vp, p32, p32]),
            "padoc_kv_pool_sync": (C.c_int, [vp, vp]),
            "padoc_kv_pool_device": (C.c_int, [vp, p32]),
            "padoc_debug_kv_pool_rehome": (C.c_int, [vp, i32]),
            "padoc_debug_set_wait_limit": (C.c_int, [C.c_uint64]),
            "padoc_branch_decode_ws_size": (C.c_int, [vp, C.POINTER(DecodeBatch), i32, C.POINTER(C.c_size_t)]),
            "padoc_branch_decode": (C.c_int, [vp, C.POINTER(DecodeBatch), i32, vp, vp, vp, vp, vp, vp, f32, vp,
                                              C.c_size_t, vp]),
            "padoc_tree_mask_build": (C.c_int, [p32, i32, C.POINTER(C.c_uint16)]),
            "padoc_depths": (C.c_int, [p32, p32, i32, p64, p64]),
            "padoc_device_status": (C.c_int, [vp]),
            "padoc_decode_plan_create": (C.c_int, [vp, C.POINTER(DecodeBatch), i32, C.POINTER(vp)]),
            "padoc_decode_plan_ws_size": (C.c_int, [vp, C.POINTER(C.c_size_t)]),
            "padoc_decode_plan_fused": (C.c_int, [vp, C.POINTER(C.c_int32)]),
            "padoc_decode_plan_upload": (C.c_int, [vp, vp, C.c_size_t, vp]),
            "padoc_decode_prefix_pass": (C.c_int, [vp, vp, f32, vp, vp]),
            "padoc_decode_own_pass": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, f32, vp, vp]),
            "padoc_decode_plan_free": (C.c_int, [vp]),
            "padoc_branch_decode_noalloc": (C.c_int, [vp, C.POINTER(DecodeBatch), i32, vp, vp, vp, vp, vp, vp, f32,
                                                      vp]),
            "padoc_verify_accept": (C.c_int, [vp, i32, i32, vp, vp, vp, i32, i32, f32, vp, vp, vp, vp]),
            "padoc_kv_commit": (C.c_int, [vp, i32, p32, p32, p32, i32, vp, vp, vp, C.c_size_t, vp]),
            "padoc_kv_reserve": (C.c_int, [vp, i32, i32]),
            "padoc_kv_advance": (C.c_int, [vp, i32, i32]),
            "padoc_kv_trim": (C.c_int, [vp, i32]),
            "padoc_sched_create": (C.c_int, [vp, C.POINTER(SchedConfig), C.POINTER(vp)]),
            "padoc_sched_destroy": (C.c_int, [vp]),
            "padoc_sched_submit": (C.c_int, [vp, i32, i64, p32]),
            "padoc_sched_schedule": (C.c_int, [vp, C.POINTER(SchedStep)]),
            "padoc_sched_update": (C.c_int, [vp, i64, i32, p32, p32, p32]),
            "padoc_sched_request": (C.c_int, [vp, i32, p32, p32, p32, p64]),
            "padoc_sched_output": (C.c_int, [vp, i32, p32, i64, p64]),
            "padoc_tree_attn_varlen_bwd_ws_size": (C.c_int, [vp, i32, C.POINTER(C.c_size_t)]),
            "padoc_tree_attn_varlen_bwd": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                     f32, vp, C.c_size_t, vp]),
            "padoc_tree_desc_bwd_plan": (C.c_int, [vp, p32, p32, p64, p64]),
            "padoc_draft_index_create": (C.c_int, [p32, p64, i32, i32, C.POINTER(vp)]),
            "padoc_draft_index_free": (C.c_int, [vp]),
            "padoc_draft_trie": (C.c_int, [vp, p32, i32, i32, i32, p32, p32, p32]),
            "padoc_draft_trie_batch": (C.c_int, [C.POINTER(vp), i32, p32, p32, i32, i32, p32, p32, p32,
                                                 C.POINTER(C.c_uint16)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(rc: int):
    if rc != OK:
        raise PadocError(rc, lib().padoc_last_error().decode(errors="replace"))


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream or None
        except Exception:
            pass
        return None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


# ------------------------------------------------------------------ tree descriptor


class TreeDesc:
    """Host descriptor of packed pages (padoc_tree_desc_build)."""

    def __init__(self, pages, order: int = PACK_CANONICAL):
        self._keep = [
            _i32([p.prefix_len for p in pages]),
            _i32([len(p.layout_len) for p in pages]),
            _i32([x for p in pages for x in p.layout_len] or [0]),
            _i32([x for p in pages for x in p.content_len] or [0]),
        ]
        spec = TreeSpec(len(pages), _p32(self._keep[0]), _p32(self._keep[1]), _p32(self._keep[2]),
                        _p32(self._keep[3]), order)
        h = C.c_void_p()
        _check(lib().padoc_tree_desc_build(C.byref(spec), C.byref(h)))
        self.handle = h

    def info(self):
        v = [C.c_int64() for _ in range(4)]
        _check(lib().padoc_tree_desc_info(self.handle, *[C.byref(x) for x in v]))
        return {"n_tokens": v[0].value, "n_qsegs": v[1].value, "n_kvsegs": v[2].value,
                "ancestor_pairs": v[3].value}

    def segments(self):
        inf = self.info()
        qs = np.zeros((max(inf["n_qsegs"], 1), 4), np.int32)
        kv = np.zeros((max(inf["n_kvsegs"], 1), 3), np.int32)
        _check(lib().padoc_tree_desc_segments(self.handle, _p32(qs), _p32(kv)))
        return qs[: inf["n_qsegs"]], kv[: inf["n_kvsegs"]]

    def bwd_plan(self):
        """Key-stationary backward plan: items [n, 4], entries [m, 5]."""
        n, m = C.c_int64(), C.c_int64()
        _check(lib().padoc_tree_desc_bwd_plan(self.handle, None, None, C.byref(n), C.byref(m)))
        it = np.zeros((max(n.value, 1), 4), np.int32)
        en = np.zeros((max(m.value, 1), 5), np.int32)
        _check(lib().padoc_tree_desc_bwd_plan(self.handle, _p32(it), _p32(en), None, None))
        return it[: n.value], en[: m.value]

    def upload(self, group: int):
        _check(lib().padoc_tree_desc_upload(self.handle, group))

    def free(self):
        if self.handle:
            lib().padoc_tree_desc_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def tree_attn_varlen(desc: TreeDesc, q, k, v, o, lse, dtype: int, Hq: int, Hkv: int, d: int,
                     scale: float = 0.0, stream=None):
    _check(lib().padoc_tree_attn_varlen(desc.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), dtype, Hq,
                                        Hkv, d, float(scale), _stream(stream)))


def tree_attn_varlen_bwd_ws_size(desc: TreeDesc, Hq: int) -> int:
    n = C.c_size_t()
    _check(lib().padoc_tree_attn_varlen_bwd_ws_size(desc.handle, Hq, C.byref(n)))
    return n.value


def tree_attn_varlen_bwd(desc: TreeDesc, q, k, v, o, lse, d_o, dq, dk, dv, dtype: int, Hq: int, Hkv: int, d: int,
                         ws, ws_bytes: int, scale: float = 0.0, stream=None):
    _check(lib().padoc_tree_attn_varlen_bwd(desc.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                                            _ptr(dq), _ptr(dk), _ptr(dv), dtype, Hq, Hkv, d, float(scale), _ptr(ws),
                                            int(ws_bytes), _stream(stream)))


# ------------------------------------------------------------------ KV pool


class KVPool:
    """Refcounted paged KV pool over caller-owned storage (padoc_kv_pool_*)."""

    def __init__(self, k_pool, v_pool, num_blocks: int, Hkv: int, d: int = 128, max_seqs: int = 1024,
                 max_blocks_per_seq: int = 512, block_size: int = 16, dtype: int = BF16):
        h = C.c_void_p()
        _check(lib().padoc_kv_pool_create(C.byref(h), _ptr(k_pool), _ptr(v_pool), num_blocks, block_size, Hkv, d,
                                          dtype, max_seqs, max_blocks_per_seq))
        self.handle = h
        self.Hkv = Hkv
        self.d = d
        self._storage = (k_pool, v_pool)

    def alloc(self, n_tokens: int = 0) -> int:
        s = C.c_int32()
        _check(lib().padoc_kv_alloc(self.handle, n_tokens, C.byref(s)))
        return s.value

    def fork(self, parent: int, fork_len: int) -> int:
        s = C.c_int32()
        _check(lib().padoc_kv_fork(self.handle, parent, fork_len, C.byref(s)))
        return s.value

    def append(self, seq: int, k, v, n: int, stream=None):
        _check(lib().padoc_kv_append(self.handle, seq, _ptr(k), _ptr(v), n, _stream(stream)))

    def release(self, seq: int):
        _check(lib().padoc_kv_release(self.handle, seq))

    def seq_info(self, seq: int):
        a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
        _check(lib().padoc_kv_seq_info(self.handle, seq, C.byref(a), C.byref(b), C.byref(c)))
        return {"length": a.value, "fork_len": b.value, "n_blocks": c.value}

    def seq_blocks(self, seq: int):
        n = self.seq_info(seq)["n_blocks"]
        out = np.zeros(max(n, 1), np.int32)
        _check(lib().padoc_kv_seq_blocks(self.handle, seq, _p32(out), len(out)))
        return out[:n]

    def refcount(self, block: int) -> int:
        r = C.c_int32()
        _check(lib().padoc_kv_block_refcount(self.handle, block, C.byref(r)))
        return r.value

    def stats(self):
        a, b = C.c_int32(), C.c_int32()
        _check(lib().padoc_kv_pool_stats(self.handle, C.byref(a), C.byref(b)))
        return {"free_blocks": a.value, "live_seqs": b.value}

    def sync(self, stream=None):
        _check(lib().padoc_kv_pool_sync(self.handle, _stream(stream)))

    def device(self) -> int:
        d = C.c_int32()
        _check(lib().padoc_kv_pool_device(self.handle, C.byref(d)))
        return d.value

    def debug_rehome(self, device: int):
        """Testing aid (padoc_debug_kv_pool_rehome): relabels the pool's device."""
        _check(lib().padoc_debug_kv_pool_rehome(self.handle, device))

    def reserve(self, seq: int, n_tokens: int):
        _check(lib().padoc_kv_reserve(self.handle, seq, n_tokens))

    def advance(self, seq: int, n: int):
        _check(lib().padoc_kv_advance(self.handle, seq, n))

    def trim(self, seq: int):
        _check(lib().padoc_kv_trim(self.handle, seq))

    def commit(self, seqs: Sequence[int], row_offsets: Sequence[int], rows: Sequence[int], n_src_rows: int,
               k_new, v_new, ws, ws_bytes: int, stream=None):
        """padoc_kv_commit: appends rows[row_offsets[i]:row_offsets[i+1]] of
        k_new / v_new to sequence seqs[i]."""
        a, b, c = _i32(seqs if len(seqs) else [0]), _i32(row_offsets if len(row_offsets) else [0]), \
            _i32(rows if len(rows) else [0])
        _check(lib().padoc_kv_commit(self.handle, len(seqs), _p32(a), _p32(b), _p32(c), n_src_rows, _ptr(k_new),
                                     _ptr(v_new), _ptr(ws), int(ws_bytes), _stream(stream)))

    def destroy(self):
        if self.handle:
            lib().padoc_kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class Batch:
    """Host arrays of one decode/verify step (padoc_decode_batch)."""

    def __init__(self, page_seq: Sequence[int], branch_offsets: Sequence[int], branch_seq: Sequence[int],
                 q_offsets: Sequence[int]):
        self._keep = [_i32(page_seq if len(page_seq) else [0]), _i32(branch_offsets), _i32(branch_seq or [0]),
                      _i32(q_offsets)]
        self.c = DecodeBatch(len(page_seq), len(branch_seq), _p32(self._keep[0]), _p32(self._keep[1]),
                             _p32(self._keep[2]), _p32(self._keep[3]))
        self.nq = int(self._keep[3][-1]) if len(branch_seq) else 0


def branch_decode_ws_size(pool: KVPool, batch: Batch, Hq: int) -> int:
    n = C.c_size_t()
    _check(lib().padoc_branch_decode_ws_size(pool.handle, C.byref(batch.c), Hq, C.byref(n)))
    return n.value


def branch_decode(pool: KVPool, batch: Batch, Hq: int, q, k_new, v_new, tree_bits, o, lse, ws, ws_bytes: int,
                  scale: float = 0.0, stream=None):
    _check(lib().padoc_branch_decode(pool.handle, C.byref(batch.c), Hq, _ptr(q), _ptr(k_new), _ptr(v_new),
                                     _ptr(tree_bits), _ptr(o), _ptr(lse), float(scale), _ptr(ws), int(ws_bytes),
                                     _stream(stream)))


def branch_decode_noalloc(pool: KVPool, batch: Batch, Hq: int, q, k_new, v_new, tree_bits, o, lse,
                          scale: float = 0.0, stream=None):
    """padoc_branch_decode with the workspace taken from the library's fixed
    device array (no device allocation; for callers that may not allocate)."""
    _check(lib().padoc_branch_decode_noalloc(pool.handle, C.byref(batch.c), Hq, _ptr(q), _ptr(k_new), _ptr(v_new),
                                             _ptr(tree_bits), _ptr(o), _ptr(lse), float(scale), _stream(stream)))


def verify_accept(logits, nq: int, vocab: int, tokens, parents, q_offsets, n_branches: int, max_nodes: int,
                  tau: float, n_acc, path, free_token, stream=None):
    """padoc_verify_accept: device arrays in, device n_acc [B], path [B, 16]
    and free_token [B] out."""
    _check(lib().padoc_verify_accept(_ptr(logits), nq, vocab, _ptr(tokens), _ptr(parents), _ptr(q_offsets),
                                     n_branches, max_nodes, float(tau), _ptr(n_acc), _ptr(path), _ptr(free_token),
                                     _stream(stream)))


class DraftIndex:
    """A request's fixed drafts with their window table (padoc_draft_index)."""

    def __init__(self, drafts: Sequence[Sequence[int]], window: int = 3):
        toks = _i32([t for d in drafts for t in d] or [0])
        offs = np.zeros(len(drafts) + 1, np.int64)
        offs[1:] = np.cumsum([len(d) for d in drafts])
        h = C.c_void_p()
        _check(lib().padoc_draft_index_create(_p32(toks), offs.ctypes.data_as(C.POINTER(C.c_int64)), len(drafts),
                                              window, C.byref(h)))
        self.handle = h

    def trie(self, accepted: Sequence[int], max_nodes: int = 16, max_depth: int = 7):
        """One step's verify block: (tokens, parents) lists."""
        acc = _i32(accepted)
        t = np.zeros(max_nodes, np.int32)
        p = np.zeros(max_nodes, np.int32)
        n = C.c_int32()
        _check(lib().padoc_draft_trie(self.handle, _p32(acc), len(acc), max_nodes, max_depth, _p32(t), _p32(p),
                                      C.byref(n)))
        return t[: n.value].tolist(), p[: n.value].tolist()

    def free(self):
        if self.handle:
            lib().padoc_draft_index_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def draft_trie_batch(indexes: Sequence[DraftIndex], accepted: Sequence[Sequence[int]], max_nodes: int = 16,
                     max_depth: int = 7):
    """padoc_draft_trie_batch: returns tokens [nq], parents [nq], q_offsets
    [B + 1] and tree bits [nq] (uint16) as numpy arrays."""
    B = len(indexes)
    hs = (C.c_void_p * max(B, 1))(*[ix.handle.value for ix in indexes])
    acc = _i32([t for a in accepted for t in a] or [0])
    aoff = np.zeros(B + 1, np.int32)
    aoff[1:] = np.cumsum([len(a) for a in accepted])
    cap = max(B * max_nodes, 1)
    t, p = np.zeros(cap, np.int32), np.zeros(cap, np.int32)
    q = np.zeros(B + 1, np.int32)
    bits = np.zeros(cap, np.uint16)
    _check(lib().padoc_draft_trie_batch(hs, B, _p32(acc), _p32(aoff), max_nodes, max_depth, _p32(t), _p32(p),
                                        _p32(q), bits.ctypes.data_as(C.POINTER(C.c_uint16))))
    nq = int(q[-1])
    return t[:nq], p[:nq], q, bits[:nq]


class Scheduler:
    """The branch scheduler over a KV pool (padoc_sched_*)."""

    STATES = ("waiting", "running", "ended", "done")

    def __init__(self, pool: "KVPool", tau: float, n_max: int, window: int, max_len: int, fork_token: int,
                 child_token: int, eos_token: int, cap: int = 4096):
        self.pool = pool
        cfg = SchedConfig(tau, n_max, window, max_len, fork_token, child_token, eos_token)
        h = C.c_void_p()
        _check(lib().padoc_sched_create(pool.handle, C.byref(cfg), C.byref(h)))
        self.handle = h
        self.cap = cap
        self._bufs = [np.zeros(cap + 1, np.int32) for _ in range(6)]

    def submit(self, prompt_len: int, arrival: int) -> int:
        r = C.c_int32()
        _check(lib().padoc_sched_submit(self.handle, prompt_len, arrival, C.byref(r)))
        return r.value

    def schedule(self):
        """admitted, preempted, and the batch as [(page_seq, [(request, seq), ...]), ...]."""
        b = self._bufs
        st = SchedStep(self.cap, 0, 0, 0, 0, *[_p32(x) for x in b])
        _check(lib().padoc_sched_schedule(self.handle, C.byref(st)))
        pages = []
        for p in range(st.n_pages):
            lo, hi = b[5][p], b[5][p + 1]
            pages.append((int(b[4][p]), [(int(b[2][i]), int(b[3][i])) for i in range(lo, hi)]))
        return b[0][: st.n_admitted].tolist(), b[1][: st.n_preempted].tolist(), pages

    def update(self, now: int, accepted):
        """accepted: [(request, [tokens...]), ...] in processing order."""
        req = _i32([r for r, _ in accepted] or [0])
        off = np.zeros(len(accepted) + 1, np.int32)
        off[1:] = np.cumsum([len(t) for _, t in accepted])
        toks = _i32([t for _, ts in accepted for t in ts] or [0])
        _check(lib().padoc_sched_update(self.handle, now, len(accepted), _p32(req), _p32(off), _p32(toks)))

    def request(self, rid: int):
        st, seq, par = C.c_int32(), C.c_int32(), C.c_int32()
        n = C.c_int64()
        _check(lib().padoc_sched_request(self.handle, rid, C.byref(st), C.byref(seq), C.byref(par), C.byref(n)))
        return {"state": self.STATES[st.value], "seq": seq.value, "parent": par.value, "n_out": n.value}

    def output(self, rid: int):
        n = C.c_int64()
        _check(lib().padoc_sched_output(self.handle, rid, None, 0, C.byref(n)))
        out = np.zeros(max(n.value, 1), np.int32)
        _check(lib().padoc_sched_output(self.handle, rid, _p32(out), len(out), C.byref(n)))
        return out[: n.value].tolist()

    def destroy(self):
        if self.handle:
            lib().padoc_sched_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class DecodePlan:
    """A planned decode step (padoc_decode_plan_*): host plan, upload, and the
    two device passes."""

    def __init__(self, pool: KVPool, batch: Batch, Hq: int):
        h = C.c_void_p()
        _check(lib().padoc_decode_plan_create(pool.handle, C.byref(batch.c), Hq, C.byref(h)))
        self.handle = h
        self._refs = (pool, batch)

    def ws_size(self) -> int:
        n = C.c_size_t()
        _check(lib().padoc_decode_plan_ws_size(self.handle, C.byref(n)))
        return n.value

    def fused(self) -> bool:
        """True when the step runs as one kernel (the prefix pass launches nothing)."""
        f = C.c_int32()
        _check(lib().padoc_decode_plan_fused(self.handle, C.byref(f)))
        return bool(f.value)

    def upload(self, ws, ws_bytes: int, stream=None):
        _check(lib().padoc_decode_plan_upload(self.handle, _ptr(ws), int(ws_bytes), _stream(stream)))

    def prefix_pass(self, q, ws, scale: float = 0.0, stream=None):
        _check(lib().padoc_decode_prefix_pass(self.handle, _ptr(q), float(scale), _ptr(ws), _stream(stream)))

    def own_pass(self, q, k_new, v_new, tree_bits, o, lse, ws, scale: float = 0.0, stream=None):
        _check(lib().padoc_decode_own_pass(self.handle, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(tree_bits),
                                           _ptr(o), _ptr(lse), float(scale), _ptr(ws), _stream(stream)))

    def free(self):
        if self.handle:
            lib().padoc_decode_plan_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


# ------------------------------------------------------------------ small helpers


def tree_mask_build(parent: Sequence[int]) -> np.ndarray:
    p = _i32(parent if len(parent) else [0])
    out = np.zeros(max(len(parent), 1), np.uint16)
    _check(lib().padoc_tree_mask_build(_p32(p), len(parent), out.ctypes.data_as(C.POINTER(C.c_uint16))))
    return out[: len(parent)]


def depths(layout_len: Sequence[int], content_len: Sequence[int]):
    a, b = _i32(list(layout_len) or [0]), _i32(list(content_len) or [0])
    s, t = C.c_int64(), C.c_int64()
    _check(lib().padoc_depths(_p32(a), _p32(b), len(layout_len), C.byref(s), C.byref(t)))
    return {"D_seq": s.value, "D_tree": t.value}


def device_status(stream=None):
    _check(lib().padoc_device_status(_stream(stream)))


def debug_set_wait_limit(ns: int):
    """Testing aid (padoc_debug_set_wait_limit): the wait limit of the
    verify own pass's keys-on-M kernel on the current device; 0 restores
    the default."""
    _check(lib().padoc_debug_set_wait_limit(int(ns)))
