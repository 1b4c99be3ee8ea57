"""ctypes binding of libns.so: argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels.  PyTorch appears here only
as device-memory and stream plumbing (``data_ptr()``, ``cuda_stream``).  When the library is
missing or cannot load, every call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libns.so")

NS_F16 = 0
NS_BF16 = 1
DTYPES = {"f16": NS_F16, "bf16": NS_BF16}

STATUS = {
    0: "NS_OK", 1: "NS_ERR_INVALID_ARG", 2: "NS_ERR_OUT_OF_MEMORY", 3: "NS_ERR_CUDA",
    4: "NS_ERR_UNSUPPORTED", 5: "NS_ERR_NOT_INITIALIZED", 6: "NS_ERR_DEVICE_CHECK",
    7: "NS_ERR_OUT_OF_BLOCKS",
}

# exported symbols declared in include/ns.h
SYMBOLS = (
    "ns_create", "ns_destroy", "ns_kv_alloc", "ns_kv_layer_ptrs", "ns_kv_prepare_step",
    "ns_kv_reserve", "ns_kv_release", "ns_kv_free_count", "ns_set_nanobatch", "ns_decode_step",
    "ns_attn_decode", "ns_linear", "ns_greedy_argmax", "ns_get_device_error",
    "ns_get_step_info", "ns_status_str", "ns_last_error_message", "ns_pool_create",
    "ns_pool_destroy", "ns_pool_prepare_step", "ns_pool_reserve", "ns_pool_release",
    "ns_pool_free_count", "ns_check_step_metadata", "ns_set_kernel_timing",
    "ns_get_kernel_timing", "ns_attn_decode_noalloc", "ns_set_token_source",
    "ns_set_graph_buckets", "ns_set_kv_offload", "ns_kv_reload", "ns_kv_save",
    "ns_pool_geometry", "ns_kv_get_pool", "ns_sched_create", "ns_sched_destroy",
    "ns_sched_add", "ns_sched_next", "ns_sched_moves", "ns_sched_commit", "ns_sched_tokens",
    "ns_sched_counts", "ns_capture_graphs", "ns_get_graph_report", "ns_attn_decode_capped",
    "ns_set_graph_chunks", "ns_sched_remove", "ns_sched_set_async", "ns_find_prompt_chunks",
    "ns_set_trace", "ns_set_gemm_cta_budget", "ns_set_step_kernel",
)


class NSError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class ModelCfg(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_layers", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_double), ("dtype", ctypes.c_int),
                ("tie_embeddings", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int), ("use_graphs", ctypes.c_int)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerWeights))]


KERNEL_KINDS = ("embed_rope", "qkv", "attention", "o_proj", "gate_up", "down", "lm_head", "other")


class KernelTiming(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int * 8), ("total_ms", ctypes.c_double * 8)]


class TraceBufs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("attn", ctypes.c_void_p), ("resid_mid", ctypes.c_void_p),
                ("resid_out", ctypes.c_void_p)]


class StepInfo(ctypes.Structure):
    _fields_ = [("kernels_per_step", ctypes.c_int), ("graphs_cached", ctypes.c_int),
                ("last_capture_ms", ctypes.c_double), ("steps", ctypes.c_longlong)]


_lib = None
_cudart = None

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float


def lib() -> ctypes.CDLL:
    """Load libns.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "ns_create": ([ctypes.POINTER(ModelCfg), ctypes.POINTER(Weights), ctypes.POINTER(P)], I),
            "ns_destroy": ([P], None),
            "ns_kv_alloc": ([P, I, I], I),
            "ns_kv_layer_ptrs": ([P, I, ctypes.POINTER(P), ctypes.POINTER(P)], I),
            "ns_kv_prepare_step": ([P, I, P, P, P], I),
            "ns_kv_reserve": ([P, I, P], I),
            "ns_kv_release": ([P, P, I], I),
            "ns_kv_free_count": ([P, ctypes.POINTER(I)], I),
            "ns_set_nanobatch": ([P, I, P, I], I),
            "ns_decode_step": ([P, I, P, P, P, P, P, P, P], I),
            "ns_attn_decode": ([P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P], I),
            "ns_linear": ([P, P, P, I, I, I, I, P], I),
            "ns_attn_decode_noalloc": ([P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P], I),
            "ns_greedy_argmax": ([P, I, I, P, P], I),
            "ns_get_device_error": ([P, ctypes.POINTER(I)], I),
            "ns_get_step_info": ([P, ctypes.POINTER(StepInfo)], I),
            "ns_status_str": ([I], ctypes.c_char_p),
            "ns_pool_create": ([I, I, I, ctypes.POINTER(P)], I),
            "ns_pool_destroy": ([P], None),
            "ns_pool_prepare_step": ([P, I, P, P, P], I),
            "ns_pool_reserve": ([P, I, P], I),
            "ns_pool_release": ([P, P, I], I),
            "ns_pool_free_count": ([P, ctypes.POINTER(I)], I),
            "ns_check_step_metadata": ([I, I, I, I, I, I, P, P, P, P, P], I),
            "ns_find_prompt_chunks": ([I, I, I, P, P, P, P, I, ctypes.POINTER(I)], I),
            "ns_last_error_message": ([], ctypes.c_char_p),
            "ns_set_kernel_timing": ([P, I], I),
            "ns_set_trace": ([P, I, ctypes.POINTER(TraceBufs)], I),
            "ns_set_gemm_cta_budget": ([P, I], I),
            "ns_set_step_kernel": ([P, I], I),
            "ns_set_token_source": ([P, P], I),
            "ns_set_graph_buckets": ([P, I, P], I),
            "ns_set_kv_offload": ([P, P, ctypes.c_size_t], I),
            "ns_kv_reload": ([P, P, I, I, P, I, P], I),
            "ns_kv_save": ([P, P, I, I, P, I, P], I),
            "ns_pool_geometry": ([P, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "ns_kv_get_pool": ([P, ctypes.POINTER(P)], I),
            "ns_sched_create": ([P, I, I, I, I, ctypes.POINTER(P)], I),
            "ns_sched_moves": ([P, P, P, P, P, I, ctypes.POINTER(I)], I),
            "ns_sched_destroy": ([P], None),
            "ns_sched_add": ([P, I, P, I, I], I),
            "ns_sched_next": ([P, P, P, P, P, P, P, P, ctypes.POINTER(I)], I),
            "ns_sched_commit": ([P, P, I, P, ctypes.POINTER(I)], I),
            "ns_sched_tokens": ([P, I, P, I, ctypes.POINTER(I)], I),
            "ns_sched_counts": ([P] + [ctypes.POINTER(I)] * 4, I),
            "ns_capture_graphs": ([P, I, P, I], I),
            "ns_set_graph_chunks": ([P, I], I),
            "ns_sched_remove": ([P, I], I),
            "ns_sched_set_async": ([P, I], I),
            "ns_attn_decode_capped": ([P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P], I),
            "ns_get_graph_report": ([P, P, I, ctypes.POINTER(I)], I),
            "ns_get_kernel_timing": ([P, ctypes.POINTER(KernelTiming)], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def check(status: int) -> None:
    if status != 0:
        raise NSError(status, lib().ns_last_error_message().decode())


def cudart() -> ctypes.CDLL:
    """The CUDA runtime libns.so links against (for plain memcpy plumbing in harnesses)."""
    global _cudart
    if _cudart is None:
        lib()
        for name in ("libcudart.so.13", "libcudart.so"):
            try:
                _cudart = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if _cudart is None:
            raise RuntimeError("libcudart not found")
        _cudart.cudaMemcpy.argtypes = [P, P, ctypes.c_size_t, I]
        _cudart.cudaMemcpy.restype = I
    return _cudart


def memcpy(dst: int, src: int, nbytes: int) -> None:
    """cudaMemcpy with cudaMemcpyDefault (direction from the pointers)."""
    r = cudart().cudaMemcpy(P(dst), P(src), ctypes.c_size_t(nbytes), 4)
    if r != 0:
        raise RuntimeError(f"cudaMemcpy failed ({r})")


def _dev(a, what: str, dtype: Optional[str] = None, min_numel: int = 0,
         itemsize: Optional[int] = None) -> Optional[int]:
    """Address of an argument the library hands to its kernels: a contiguous CUDA tensor (of
    torch dtype ``dtype``, or of ``itemsize``-byte elements, and at least ``min_numel``
    elements, where given) or a raw device address (an int, the caller's responsibility).  Host
    memory, a buffer of the wrong element type or a short buffer would be dereferenced on the
    device, so it is refused here, before anything is launched, with the library's own
    INVALID_ARG status."""
    if a is None or isinstance(a, int):
        return a
    if isinstance(a, np.ndarray) or not getattr(a, "is_cuda", False):
        raise NSError(1, f"{what} must be device memory (a CUDA tensor or a device address)")
    if dtype is not None and str(a.dtype) != "torch." + dtype:
        raise NSError(1, f"{what} must be {dtype}, not {a.dtype}")
    if itemsize is not None and a.element_size() != itemsize:
        raise NSError(1, f"{what} must have {itemsize}-byte elements, not {a.element_size()}")
    if a.numel() < min_numel:
        raise NSError(1, f"{what} has {a.numel()} elements, needs at least {min_numel}")
    return _ptr(a)


def _same_rows(batch: int, **arrays) -> None:
    """Host metadata arrays must all describe ``batch`` rows (the library reads that many)."""
    for name, a in arrays.items():
        if a is not None and (a.ndim < 1 or a.shape[0] != batch):
            raise NSError(1, f"{name} has {a.shape[0] if a.ndim else 0} rows, the batch is {batch}")


def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("host arrays must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return a.data_ptr()
    raise TypeError(type(a))


def _stream(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class GraphInfo(ctypes.Structure):
    _fields_ = [("batch", I), ("n_split", I), ("attn_cta_budget", I), ("with_lm", I),
                ("chunk_rows", I), ("kv_offload", I), ("kernels", I), ("capture_ms", ctypes.c_double),
                ("gemm_cta_budget", I), ("attn_queue", I)]


class DecodeStep:
    """A model handle: ns_create / ns_kv_alloc / ns_decode_step and friends.

    ``weights`` is a dict shaped like ``synth.model_weights`` (host numpy arrays or device
    tensors, storage dtype); the library copies them.
    """

    def __init__(self, shape, weights, max_batch: int, max_blocks_per_seq: int,
                 use_graphs: bool = True):
        L = lib()
        self.shape = shape
        self.max_batch = max_batch
        self.mb = max_blocks_per_seq
        cfg = ModelCfg(shape.hidden, shape.n_layers, shape.n_q_heads, shape.n_kv_heads,
                       shape.head_dim, shape.ffn, shape.vocab, float(shape.rms_eps),
                       float(shape.rope_theta), DTYPES[shape.dtype],
                       1 if shape.tie_embeddings else 0, max_batch, max_blocks_per_seq,
                       1 if use_graphs else 0)
        keep = []
        layers = (LayerWeights * shape.n_layers)()
        for l, lw in enumerate(weights["layers"]):
            for k in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
                a = lw[k]
                if isinstance(a, np.ndarray):
                    a = np.ascontiguousarray(a)
                keep.append(a)
                setattr(layers[l], k, _ptr(a))
        emb = np.ascontiguousarray(weights["embed"]) if isinstance(weights["embed"], np.ndarray) else weights["embed"]
        fin = np.ascontiguousarray(weights["final_norm"]) if isinstance(weights["final_norm"], np.ndarray) else weights["final_norm"]
        head = weights.get("lm_head")
        keep += [emb, fin, head]
        w = Weights(_ptr(emb), _ptr(fin), _ptr(head), layers)
        h = P()
        check(L.ns_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)))
        self.h = h
        self.num_blocks = 0
        self.block_size = 0

    def close(self) -> None:
        if getattr(self, "h", None):
            lib().ns_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_alloc(self, num_blocks: int, block_size: int = 16) -> None:
        check(lib().ns_kv_alloc(self.h, num_blocks, block_size))
        self.num_blocks = num_blocks
        self.block_size = block_size

    def kv_layer_ptrs(self, layer: int):
        k, v = P(), P()
        check(lib().ns_kv_layer_ptrs(self.h, layer, ctypes.byref(k), ctypes.byref(v)))
        return k.value, v.value

    def kv_pool_bytes(self) -> int:
        s = self.shape
        return self.num_blocks * s.n_kv_heads * self.block_size * s.head_dim * 2

    def prepare_step(self, positions: np.ndarray, block_tables: np.ndarray) -> np.ndarray:
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        assert block_tables.dtype == np.int32 and block_tables.flags["C_CONTIGUOUS"]
        slots = np.zeros(pos.shape[0], dtype=np.int64)
        check(lib().ns_kv_prepare_step(self.h, pos.shape[0], _ptr(pos), _ptr(block_tables),
                                       _ptr(slots)))
        return slots

    def reserve(self, n: int) -> np.ndarray:
        out = np.zeros(max(n, 1), dtype=np.int32)
        check(lib().ns_kv_reserve(self.h, n, _ptr(out)))
        return out[:n]

    def release(self, ids: Sequence[int]) -> None:
        a = np.ascontiguousarray(ids, dtype=np.int32)
        check(lib().ns_kv_release(self.h, _ptr(a) if a.size else None, a.size))

    def free_count(self) -> int:
        n = I()
        check(lib().ns_kv_free_count(self.h, ctypes.byref(n)))
        return n.value

    def set_nanobatch(self, sizes: Optional[Sequence[int]] = None, attn_cta_budget: int = 0,
                      gemm_cta_budget: int = 0):
        """Nano-batch split (None: unsplit) with the attention and persistent-GEMM CTA caps of
        its nano-ops (0: none)."""
        check(lib().ns_set_gemm_cta_budget(self.h, gemm_cta_budget))
        if not sizes or len(sizes) == 1:
            check(lib().ns_set_nanobatch(self.h, 1, None, attn_cta_budget))
            return
        a = np.ascontiguousarray(sizes, dtype=np.int32)
        check(lib().ns_set_nanobatch(self.h, a.size, _ptr(a), attn_cta_budget))

    def set_step_kernel(self, mode: int) -> None:
        """0: one kernel per stage; 1: steps of at most 32 decode rows as one persistent kernel
        (ns_set_step_kernel)."""
        check(lib().ns_set_step_kernel(self.h, int(mode)))

    def step(self, token_ids, positions, block_tables, seq_lens, slot_mapping, logits,
             stream=None) -> None:
        """One decode step; host metadata arrays, ``logits`` a device fp32 [B, V] buffer
        (None: stop after the last layer, no LM head).  ``token_ids`` may be None after
        ``set_token_source``."""
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        tok = None if token_ids is None else np.ascontiguousarray(token_ids, dtype=np.int32)
        tab = np.ascontiguousarray(block_tables, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        slot = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        if tab.ndim != 2 or tab.shape[1] != self.mb:
            raise ValueError(f"block_tables must be [batch, {self.mb}]")
        B = pos.shape[0] if pos.ndim == 1 else -1
        _same_rows(B, token_ids=tok, block_tables=tab, seq_lens=sl, slot_mapping=slot)
        out = _dev(logits, "logits", "float32", B * self.shape.vocab)
        check(lib().ns_decode_step(self.h, B, _ptr(tok), _ptr(pos), _ptr(tab),
                                   _ptr(sl), _ptr(slot), out, _stream(stream)))

    def device_error(self) -> int:
        c = I()
        check(lib().ns_get_device_error(self.h, ctypes.byref(c)))
        return c.value

    def set_graph_buckets(self, sizes: Optional[Sequence[int]] = None) -> None:
        """Replay graphs captured for these batch sizes only, padding smaller batches."""
        a = np.ascontiguousarray(sizes or [], dtype=np.int32)
        check(lib().ns_set_graph_buckets(self.h, a.size, _ptr(a) if a.size else None))

    def set_graph_chunks(self, capture: bool) -> None:
        """False: steps with prompt chunks launch eagerly; only decode-only steps use graphs."""
        check(lib().ns_set_graph_chunks(self.h, 1 if capture else 0))

    def set_token_source(self, device_ids=None) -> None:
        """Read token ids from a device int32 buffer (e.g. the previous argmax) or, with None,
        from the host arrays passed to ``step``."""
        # any row may name any entry (token id -(r + 1)), so the buffer holds max_batch ids
        check(lib().ns_set_token_source(self.h, _dev(device_ids, "device_ids", "int32",
                                                     self.max_batch)))

    def pool(self) -> int:
        """The handle's block pool (borrowed), for ``BatchFormer``."""
        out = P()
        check(lib().ns_kv_get_pool(self.h, ctypes.byref(out)))
        return out.value

    def kv_row_elems(self) -> int:
        """Elements of one (layer, token) K/V row of the offload layout: K then V."""
        return 2 * self.shape.n_kv_heads * self.shape.head_dim

    def set_kv_offload(self, host_buf=None) -> None:
        """Mirror each step's new K/V into ``host_buf``, pinned host memory of
        [n_layers][max_batch][kv_row_elems] storage-dtype elements (e.g. a pinned torch tensor),
        or stop with None."""
        if host_buf is None:
            check(lib().ns_set_kv_offload(self.h, None, 0))
            return
        nbytes = host_buf.numel() * host_buf.element_size() if hasattr(host_buf, "numel") else host_buf.nbytes
        check(lib().ns_set_kv_offload(self.h, _ptr(host_buf), nbytes))

    def _kv_transfer(self, fn, buf, n_tokens: int, first_pos: int, block_table, stream) -> None:
        tab = np.ascontiguousarray(block_table, dtype=np.int32)
        nbytes = buf.numel() * buf.element_size() if hasattr(buf, "numel") else buf.nbytes
        if nbytes < self.shape.n_layers * n_tokens * self.kv_row_elems() * 2:
            raise ValueError("buffer smaller than [n_layers][n_tokens][kv_row_elems]")
        check(fn(self.h, _ptr(buf), n_tokens, first_pos, _ptr(tab), tab.size, _stream(stream)))

    def kv_reload(self, host_src, n_tokens: int, first_pos: int, block_table, stream=None) -> None:
        """Scatter [n_layers][n_tokens][kv_row_elems] host K/V rows of positions first_pos..
        into the pages of ``block_table``."""
        self._kv_transfer(lib().ns_kv_reload, host_src, n_tokens, first_pos, block_table, stream)

    def kv_save(self, host_dst, n_tokens: int, first_pos: int, block_table, stream=None) -> None:
        """Gather the K/V of positions first_pos.. of ``block_table`` into host rows."""
        self._kv_transfer(lib().ns_kv_save, host_dst, n_tokens, first_pos, block_table, stream)

    def set_trace(self, layer: int, q=None, attn=None, resid_mid=None, resid_out=None) -> None:
        """Copy layer ``layer``'s q (after RoPE), attention output, residual after the attention
        block and residual after the layer into these device buffers during the next eager
        steps (graphs are bypassed); ``layer`` < 0 turns the trace off."""
        if layer < 0:
            check(lib().ns_set_trace(self.h, -1, None))
            return
        B, s = self.max_batch, self.shape
        qd = s.n_q_heads * s.head_dim
        tb = TraceBufs(_dev(q, "q", None, B * qd, 2), _dev(attn, "attn", None, B * qd, 2),
                       _dev(resid_mid, "resid_mid", "float32", B * s.hidden),
                       _dev(resid_out, "resid_out", "float32", B * s.hidden))
        check(lib().ns_set_trace(self.h, layer, ctypes.byref(tb)))

    def set_kernel_timing(self, on: bool) -> None:
        check(lib().ns_set_kernel_timing(self.h, 1 if on else 0))

    def kernel_timing(self) -> dict:
        t = KernelTiming()
        check(lib().ns_get_kernel_timing(self.h, ctypes.byref(t)))
        return {KERNEL_KINDS[i]: (t.launches[i], t.total_ms[i]) for i in range(8)
                if t.launches[i] > 0}

    def capture_graphs(self, sizes: Sequence[int], with_lm: bool = True) -> None:
        """Capture the decode-only graphs of these batch sizes now (start-up)."""
        a = np.ascontiguousarray(sizes, dtype=np.int32)
        check(lib().ns_capture_graphs(self.h, a.size, _ptr(a) if a.size else None, 1 if with_lm else 0))

    def graph_report(self) -> list:
        """One dict per captured graph: batch, n_split, attn_cta_budget, with_lm, chunk_rows,
        kv_offload, kernels, capture_ms, gemm_cta_budget, attn_queue."""
        n = I()
        check(lib().ns_get_graph_report(self.h, None, 0, ctypes.byref(n)))
        arr = (GraphInfo * max(n.value, 1))()
        check(lib().ns_get_graph_report(self.h, arr, n.value, ctypes.byref(n)))
        return [{f: getattr(arr[i], f) for f, _ in GraphInfo._fields_} for i in range(n.value)]

    def info(self) -> StepInfo:
        s = StepInfo()
        check(lib().ns_get_step_info(self.h, ctypes.byref(s)))
        return s


def _attn_args(q, k_pool, v_pool, block_tables, seq_lens, out, n_q_heads, n_kv_heads,
               head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype):
    """The C arguments shared by the attention calls, each device buffer checked against the
    sizes the kernel reads or writes: q and out [batch][n_q_heads][head_dim] and the pools
    [num_blocks][n_kv_heads][block_size][head_dim] of 16-bit elements, block_tables int32
    [batch][max_blocks_per_seq], seq_lens int32 [batch]."""
    batch = int(seq_lens.shape[0])
    rows = batch * n_q_heads * head_dim
    pool = num_blocks * n_kv_heads * block_size * head_dim
    return (_dev(q, "q", None, rows, 2), _dev(k_pool, "k_pool", None, pool, 2),
            _dev(v_pool, "v_pool", None, pool, 2),
            _dev(block_tables, "block_tables", "int32", batch * max_blocks_per_seq),
            _dev(seq_lens, "seq_lens", "int32", batch), _dev(out, "out", None, rows, 2),
            batch, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
            float(scale), DTYPES[dtype])


def attn_decode(q, k_pool, v_pool, block_tables, seq_lens, out, n_q_heads: int,
                n_kv_heads: int, head_dim: int, block_size: int, max_blocks_per_seq: int,
                num_blocks: int, scale: float, dtype: str, stream=None, cta_budget: int = 0) -> None:
    """Paged decode attention; ``cta_budget`` > 0 caps its CTAs (ns_attn_decode_capped)."""
    args = _attn_args(q, k_pool, v_pool, block_tables, seq_lens, out, n_q_heads, n_kv_heads,
                      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype)
    if cta_budget:
        check(lib().ns_attn_decode_capped(*args, cta_budget, _stream(stream)))
    else:
        check(lib().ns_attn_decode(*args, _stream(stream)))


def attn_decode_noalloc(q, k_pool, v_pool, block_tables, seq_lens, out, n_q_heads: int,
                        n_kv_heads: int, head_dim: int, block_size: int,
                        max_blocks_per_seq: int, num_blocks: int, scale: float, dtype: str,
                        dev_err=None, stream=None) -> None:
    """The allocation-free attention call (fixed in-library scratch; see include/ns.h)."""
    args = _attn_args(q, k_pool, v_pool, block_tables, seq_lens, out, n_q_heads, n_kv_heads,
                      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype)
    check(lib().ns_attn_decode_noalloc(*args, _dev(dev_err, "dev_err", "int32", 1),
                                       _stream(stream)))


def linear(w, x, y, m: int, n: int, k: int, dtype: str, stream=None) -> None:
    """y[m][n] (fp32) = x[m][k] . w[n][k]^T on the projection kernel (16-bit w and x)."""
    check(lib().ns_linear(_dev(w, "w", None, n * k, 2), _dev(x, "x", None, m * k, 2),
                          _dev(y, "y", "float32", m * n), m, n, k, DTYPES[dtype],
                          _stream(stream)))


def greedy_argmax(logits, out_ids, stream=None) -> None:
    b, v = int(logits.shape[0]), int(logits.shape[1])
    check(lib().ns_greedy_argmax(_dev(logits, "logits", "float32"), b, v,
                                 _dev(out_ids, "out_ids", "int32", b), _stream(stream)))


def device_error() -> int:
    c = I()
    check(lib().ns_get_device_error(None, ctypes.byref(c)))
    return c.value


class BlockPool:
    """Host-only block pool (ns_pool_*): the allocator and slot mapper, no GPU needed."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        h = P()
        check(lib().ns_pool_create(num_blocks, block_size, max_blocks_per_seq, ctypes.byref(h)))
        self.h = h
        self.mb = max_blocks_per_seq

    def close(self):
        if getattr(self, "h", None):
            lib().ns_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prepare_step(self, positions, block_tables) -> np.ndarray:
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        assert block_tables.dtype == np.int32 and block_tables.flags["C_CONTIGUOUS"]
        slots = np.zeros(max(pos.shape[0], 1), dtype=np.int64)
        check(lib().ns_pool_prepare_step(self.h, pos.shape[0], _ptr(pos), _ptr(block_tables),
                                         _ptr(slots)))
        return slots[: pos.shape[0]]

    def reserve(self, n: int) -> np.ndarray:
        out = np.zeros(max(n, 1), dtype=np.int32)
        check(lib().ns_pool_reserve(self.h, n, _ptr(out)))
        return out[:n]

    def release(self, ids) -> None:
        a = np.ascontiguousarray(ids, dtype=np.int32)
        check(lib().ns_pool_release(self.h, _ptr(a) if a.size else None, a.size))

    def free_count(self) -> int:
        n = I()
        check(lib().ns_pool_free_count(self.h, ctypes.byref(n)))
        return n.value


def check_step_metadata(num_blocks, block_size, max_blocks_per_seq, vocab, max_batch,
                        token_ids, positions, block_tables, seq_lens, slot_mapping) -> int:
    """Run the library's host validation; returns the ns_status code (0 = valid)."""
    tok = np.ascontiguousarray(token_ids, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    tab = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    slot = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    try:
        _same_rows(pos.shape[0] if pos.ndim == 1 else -1, token_ids=tok, block_tables=tab,
                   seq_lens=sl, slot_mapping=slot)
    except NSError as e:
        return e.status
    if tab.ndim != 2 or tab.shape[1] != max_blocks_per_seq:
        return 1
    return lib().ns_check_step_metadata(num_blocks, block_size, max_blocks_per_seq, vocab,
                                        max_batch, tok.shape[0], _ptr(tok), _ptr(pos),
                                        _ptr(tab), _ptr(sl), _ptr(slot))


def find_prompt_chunks(block_size: int, positions, block_tables, seq_lens) -> list:
    """First rows of the prompt chunks ns_decode_step attends with the causal chunk kernel."""
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    tab = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = pos.shape[0] if pos.ndim == 1 else -1
    _same_rows(B, block_tables=tab, seq_lens=sl)
    if tab.ndim != 2:
        raise NSError(1, "block_tables must be [batch, max_blocks_per_seq]")
    out = np.zeros(max(B, 1), dtype=np.int32)
    n = I()
    check(lib().ns_find_prompt_chunks(block_size, tab.shape[1], B, _ptr(pos), _ptr(tab), _ptr(sl),
                                      _ptr(out), out.size, ctypes.byref(n)))
    return out[:n.value].tolist()


class BatchFormer:
    """Constant-dense-batch former (ns_sched_*): decode rows first, then prompt chunks up to
    ``dense_tokens`` rows per step.  ``pool`` is a ``BlockPool`` or ``DecodeStep.pool()``."""

    def __init__(self, pool, dense_tokens: int, max_blocks_per_seq: int, eos_token: int,
                 predicted_new_tokens: int = 0):
        self._pool = pool  # keeps a BlockPool alive
        ph = pool.h if isinstance(pool, BlockPool) else P(pool)
        h = P()
        check(lib().ns_sched_create(ph, dense_tokens, max_blocks_per_seq, eos_token,
                                    predicted_new_tokens, ctypes.byref(h)))
        self.h, self.D, self.mb = h, dense_tokens, max_blocks_per_seq

    def close(self):
        if getattr(self, "h", None):
            lib().ns_sched_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, request_id: int, prompt, max_new_tokens: int) -> None:
        a = np.ascontiguousarray(prompt, dtype=np.int32)
        check(lib().ns_sched_add(self.h, request_id, _ptr(a) if a.size else None, a.size, max_new_tokens))

    def next(self) -> dict:
        """The next step's rows: token_ids, positions, block_tables, seq_lens, slot_mapping,
        row_request, row_samples (host arrays of the step's row count)."""
        D, mb = self.D, self.mb
        out = {"token_ids": np.zeros(D, np.int32), "positions": np.zeros(D, np.int32),
               "block_tables": np.zeros((D, mb), np.int32), "seq_lens": np.zeros(D, np.int32),
               "slot_mapping": np.zeros(D, np.int64), "row_request": np.zeros(D, np.int32),
               "row_samples": np.zeros(D, np.int32)}
        n = I()
        check(lib().ns_sched_next(self.h, *(_ptr(out[k]) for k in (
            "token_ids", "positions", "block_tables", "seq_lens", "slot_mapping", "row_request",
            "row_samples")), ctypes.byref(n)))
        return {k: v[:n.value] for k, v in out.items()}

    def moves(self) -> list:
        """The formed step's moves, saves first: (kind, request id, n_tokens, block ids);
        kind 0 = save the cached tokens from those blocks, 1 = reload them into them."""
        n = I()
        check(lib().ns_sched_moves(self.h, None, None, None, None, 0, ctypes.byref(n)))
        m = n.value
        k, r, t = (np.zeros(max(m, 1), np.int32) for _ in range(3))
        tab = np.zeros((max(m, 1), self.mb), np.int32)
        check(lib().ns_sched_moves(self.h, _ptr(k), _ptr(r), _ptr(t), _ptr(tab), m, ctypes.byref(n)))
        bs = self._block_size()
        return [(int(k[i]), int(r[i]), int(t[i]), tab[i, :(int(t[i]) + bs - 1) // bs].copy())
                for i in range(m)]

    def _block_size(self) -> int:
        nb, bs = I(), I()
        ph = self._pool.h if isinstance(self._pool, BlockPool) else P(self._pool)
        check(lib().ns_pool_geometry(ph, ctypes.byref(nb), ctypes.byref(bs)))
        return bs.value

    def commit(self, sampled) -> list:
        a = np.ascontiguousarray(sampled, dtype=np.int32)
        fin = np.zeros(max(a.size, 1), np.int32)
        n = I()
        check(lib().ns_sched_commit(self.h, _ptr(a) if a.size else None, a.size, _ptr(fin), ctypes.byref(n)))
        return fin[:n.value].tolist()

    def tokens(self, request_id: int) -> list:
        n = I()
        check(lib().ns_sched_tokens(self.h, request_id, None, 0, ctypes.byref(n)))
        out = np.zeros(max(n.value, 1), np.int32)
        check(lib().ns_sched_tokens(self.h, request_id, _ptr(out), n.value, ctypes.byref(n)))
        return out[:n.value].tolist()

    def remove(self, request_id: int) -> None:
        """Forget a finished request."""
        check(lib().ns_sched_remove(self.h, request_id))

    def set_async(self, on: bool) -> None:
        """Form the next step before the previous one is committed (tokens not yet on the host
        are written -(row + 1): the previous step's sampled token at that row)."""
        check(lib().ns_sched_set_async(self.h, 1 if on else 0))

    def counts(self):
        """(requests with prompt left, running, preempted, finished and not removed)."""
        w, r, p, f = I(), I(), I(), I()
        check(lib().ns_sched_counts(self.h, ctypes.byref(w), ctypes.byref(r), ctypes.byref(p),
                                    ctypes.byref(f)))
        return w.value, r.value, p.value, f.value
