"""Python binding of libtq_gb300.so, the C ABI declared in include/tq_kv.h.

Argument marshalling only: every step of the store and decode path runs in the
library's CUDA kernels.  Device buffers are torch tensors owned by the caller
(or by :class:`TQCache`, a convenience owner); PyTorch provides memory and
streams, nothing else.  The library must have been built
(``python -m turboquant_bit_kv_tq_gb300._build`` or ``__graft_entry__.build()``);
importing the functions works without it, calling them raises.
"""

import ctypes
import os

import numpy as np

__all__ = [
    "TQError", "tq_cache_config", "TQ_DTYPE_F32", "TQ_DTYPE_BF16", "TQ_OUT_ROTATED", "TQ_V_MSE", "TQ_V_G32",
    "TQ_CODEBOOK_LLOYD", "TQ_CODEBOOK_UNIFORM", "tq_make_uniform_codebook",
    "TQ_DEVERR_SLOT", "TQ_DEVERR_BLOCK", "TQ_DEVERR_SEQLEN", "TQ_DEVERR_TAIL", "TQ_DEVERR_TIMEOUT", "EXPORTED",
    "library_path", "load_library", "tq_status_string", "tq_last_cuda_error", "tq_make_codebook",
    "tq_make_rotation_signs",
    "tq_make_qjl_matrix", "tq_cache_sizes", "tq_cache_create", "tq_cache_destroy", "tq_cache_export_params",
    "tq_store", "tq_decode_attention", "tq_decode_attention_noalloc", "tq_set_profile_events",
    "tq_get_device_error", "tq_set_store_small_max", "tq_extend_attention", "TQ_DEVERR_CHUNK", "TQCache",
    "TQ_PROF_STORE", "TQ_PROF_DECODE_SPLIT", "tq_check_wait_timeout", "tq_store_decode_attention",
]

TQ_DTYPE_F32, TQ_DTYPE_BF16 = 0, 1
TQ_OUT_ROTATED = 0x100
TQ_V_MSE, TQ_V_G32 = 0, 1
TQ_CODEBOOK_LLOYD, TQ_CODEBOOK_UNIFORM = 0, 1
TQ_DEVERR_SLOT, TQ_DEVERR_BLOCK, TQ_DEVERR_SEQLEN, TQ_DEVERR_TAIL = 1, 2, 4, 8
TQ_DEVERR_TIMEOUT, TQ_DEVERR_CHUNK = 16, 32

# every function include/tq_kv.h declares
EXPORTED = [
    "tq_status_string", "tq_make_codebook", "tq_make_rotation_signs", "tq_make_qjl_matrix", "tq_cache_sizes",
    "tq_cache_create", "tq_cache_destroy", "tq_cache_export_params", "tq_store", "tq_decode_attention",
    "tq_set_profile_events", "tq_get_device_error", "tq_decode_attention_noalloc", "tq_last_cuda_error",
    "tq_set_store_small_max", "tq_make_uniform_codebook", "tq_extend_attention", "tq_check_wait_timeout",
    "tq_store_decode_attention",
]
TQ_PROF_STORE, TQ_PROF_DECODE_SPLIT = 0, 1


class TQError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = f"{what}: {tq_status_string(status)} ({status})"
        if status == -4:
            msg += f" [{tq_last_cuda_error()}]"
        super().__init__(msg)


class tq_cache_config(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
        ("k_bits", ctypes.c_int32),
        ("k_qjl", ctypes.c_int32),
        ("v_mode", ctypes.c_int32),
        ("v_bits", ctypes.c_int32),
        ("seed_rot", ctypes.c_uint64),
        ("seed_qjl", ctypes.c_uint64),
        ("max_batch", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("split_blocks", ctypes.c_int32),
        ("tail_cap", ctypes.c_int32),
        ("k_codebook", ctypes.c_int32),
        ("v_codebook", ctypes.c_int32),
    ]

    def __init__(self, **kw):
        defaults = dict(block_size=16, k_qjl=1, seed_rot=2, seed_qjl=1, max_batch=1, split_blocks=32, tail_cap=0)
        defaults.update(kw)
        super().__init__(**defaults)


_LIB = None
_P = ctypes.c_void_p


def library_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtq_gb300.so")


def load_library():
    """Load libtq_gb300.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -m turboquant_bit_kv_tq_gb300._build)")
        lib = ctypes.CDLL(path)
        i32, i64, u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
        dp = ctypes.POINTER(ctypes.c_double)
        cfgp = ctypes.POINTER(tq_cache_config)
        sz = ctypes.POINTER(ctypes.c_size_t)
        sig = {
            "tq_status_string": (ctypes.c_char_p, [i32]),
            "tq_last_cuda_error": (ctypes.c_char_p, []),
            "tq_make_codebook": (i32, [i32, i32, dp, dp, dp]),
            "tq_make_uniform_codebook": (i32, [i32, i32, dp, dp, dp]),
            "tq_make_rotation_signs": (i32, [i32, u64, ctypes.POINTER(ctypes.c_float)]),
            "tq_make_qjl_matrix": (i32, [i32, u64, ctypes.POINTER(ctypes.c_uint16)]),
            "tq_cache_sizes": (i32, [cfgp, sz, sz, sz, sz]),
            "tq_cache_create": (i32, [cfgp, _P, _P, _P, ctypes.POINTER(_P)]),
            "tq_cache_destroy": (i32, [_P]),
            "tq_cache_export_params": (i32, [_P, _P, _P, _P, _P, _P, _P]),
            "tq_store": (i32, [_P, _P, _P, i32, i64, _P, _P, _P]),
            "tq_decode_attention": (i32, [_P, _P, i32, _P, _P, _P, _P, _P, _P, ctypes.c_float, i32, _P, i32, _P]),
            "tq_set_profile_events": (i32, [_P, i32, _P, _P]),
            "tq_extend_attention": (i32, [_P, _P, i32, _P, _P, _P, _P, _P, _P, ctypes.c_float, i32, i32, _P, i32, _P]),
            "tq_decode_attention_noalloc": (
                i32, [_P, _P, i32, _P, _P, _P, _P, _P, _P, ctypes.c_float, i32, _P, i32, _P]),
            "tq_get_device_error": (i32, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
            "tq_set_store_small_max": (i32, [i64]),
            "tq_check_wait_timeout": (i32, [_P, ctypes.c_uint32, _P]),
            "tq_store_decode_attention": (
                i32, [_P, _P, _P, i32, i64, _P, _P, i32, _P, _P, _P, _P, _P, _P, ctypes.c_float, i32, _P, i32, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _LIB = lib
    return _LIB


def _check(status, what):
    if status != 0:
        raise TQError(status, what)


def tq_status_string(status):
    return load_library().tq_status_string(status).decode()


def tq_last_cuda_error():
    """The CUDA runtime message behind the last TQ_ERR_CUDA on this thread."""
    return load_library().tq_last_cuda_error().decode()


def tq_set_store_small_max(max_vectors):
    """Largest store (in token x KV-head vectors) encoded one vector per CTA;
    negative restores the default (16 x the SM count)."""
    _check(load_library().tq_set_store_small_max(int(max_vectors)), "tq_set_store_small_max")


def _dptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def tq_make_codebook(d, bits):
    """(centroids [2^bits], boundaries [2^bits-1], per-vector mse) as float64."""
    c = np.zeros(2**bits)
    b = np.zeros(2**bits - 1)
    mse = ctypes.c_double()
    _check(load_library().tq_make_codebook(d, bits, _dptr(c), _dptr(b), ctypes.byref(mse)), "tq_make_codebook")
    return c, b, mse.value


def tq_make_uniform_codebook(d, bits):
    """Uniform-grid (centroids, boundaries, per-vector mse) as float64."""
    c = np.zeros(2**bits)
    b = np.zeros(2**bits - 1)
    mse = ctypes.c_double()
    _check(load_library().tq_make_uniform_codebook(d, bits, _dptr(c), _dptr(b), ctypes.byref(mse)),
           "tq_make_uniform_codebook")
    return c, b, mse.value


def tq_make_rotation_signs(d, seed):
    out = np.zeros(d, np.float32)
    _check(load_library().tq_make_rotation_signs(d, seed, out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))),
           "tq_make_rotation_signs")
    return out


def tq_make_qjl_matrix(d, seed):
    """S as bfloat16 bit patterns, uint16 [d, d] (row j = output j)."""
    out = np.zeros((d, d), np.uint16)
    _check(load_library().tq_make_qjl_matrix(d, seed, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "tq_make_qjl_matrix")
    return out


def tq_cache_sizes(cfg):
    vals = [ctypes.c_size_t() for _ in range(4)]
    _check(load_library().tq_cache_sizes(ctypes.byref(cfg), *[ctypes.byref(v) for v in vals]), "tq_cache_sizes")
    return dict(zip(["page_bytes", "cache_bytes", "params_bytes", "workspace_bytes"], [v.value for v in vals]))


def _stream_ptr(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def tq_cache_create(cfg, params, workspace, stream=None):
    h = _P()
    _check(load_library().tq_cache_create(ctypes.byref(cfg), _P(params.data_ptr()), _P(workspace.data_ptr()),
                                          _stream_ptr(stream), ctypes.byref(h)), "tq_cache_create")
    return h


def tq_cache_destroy(handle):
    _check(load_library().tq_cache_destroy(handle), "tq_cache_destroy")


def tq_cache_export_params(handle, cfg):
    d = cfg.head_dim
    out = dict(signs=np.zeros(d, np.float32), qjl_bf16=np.zeros((d, d), np.uint16),
               k_centroids=np.zeros(2**cfg.k_bits), k_boundaries=np.zeros(2**cfg.k_bits - 1))
    if cfg.v_mode == TQ_V_MSE:
        out.update(v_centroids=np.zeros(2**cfg.v_bits), v_boundaries=np.zeros(2**cfg.v_bits - 1))
    p = lambda k: _P(out[k].ctypes.data) if k in out else _P()  # noqa: E731
    _check(load_library().tq_cache_export_params(handle, p("signs"), p("qjl_bf16"), p("k_centroids"),
                                                 p("k_boundaries"), p("v_centroids"), p("v_boundaries")),
           "tq_cache_export_params")
    return out


def _dtype_code(t):
    import torch

    if t.dtype == torch.float32:
        return TQ_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return TQ_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def _dev(t, name, dtype=None):
    if t is None:
        return _P()
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return _P(t.data_ptr())


def tq_store(handle, k, v, slot_mapping, cache, stream=None):
    """k, v [T, H_kv, d] (f32 or bf16, same dtype); slot_mapping int64 [T]."""
    import torch

    if k.dtype != v.dtype or k.shape != v.shape:
        raise ValueError("k and v must have the same shape and dtype")
    _check(load_library().tq_store(handle, _dev(k, "k"), _dev(v, "v"), _dtype_code(k), k.shape[0],
                                   _dev(slot_mapping, "slot_mapping", torch.int64), _dev(cache, "cache"),
                                   _stream_ptr(stream)), "tq_store")


def tq_decode_attention(handle, q, cache, block_table, seq_lens, out, tail_k=None, tail_v=None, tail_lens=None,
                        scale=0.0, stream=None, rotated=False):
    """q [B, H_q, d] (f32/bf16); block_table int32 [B, max_blocks_per_seq];
    seq_lens int32 [B]; out [B, H_q, d] (f32/bf16); optional bf16 tail;
    rotated: MSE values only, out in the rotated space (R out)."""
    import torch

    if tail_k is not None:
        _dev(tail_k, "tail_k", torch.bfloat16)
        _dev(tail_v, "tail_v", torch.bfloat16)
    _check(load_library().tq_decode_attention(
        handle, _dev(q, "q"), _dtype_code(q), _dev(cache, "cache"), _dev(block_table, "block_table", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), _dev(tail_k, "tail_k"), _dev(tail_v, "tail_v"),
        _dev(tail_lens, "tail_lens", torch.int32), float(scale), q.shape[0], _dev(out, "out"),
        _dtype_code(out) | (TQ_OUT_ROTATED if rotated else 0), _stream_ptr(stream)), "tq_decode_attention")


def tq_store_decode_attention(handle, k, v, slot_mapping, q, cache, block_table, seq_lens, out, tail_k=None,
                              tail_v=None, tail_lens=None, scale=0.0, stream=None, rotated=False):
    """tq_store(k, v, slot_mapping) then tq_decode_attention(q, ...) in one
    call; k and v may have zero tokens (nothing is stored)."""
    import torch

    if k.dtype != v.dtype or k.shape != v.shape:
        raise ValueError("k and v must have the same shape and dtype")
    if tail_k is not None:
        _dev(tail_k, "tail_k", torch.bfloat16)
        _dev(tail_v, "tail_v", torch.bfloat16)
    _check(load_library().tq_store_decode_attention(
        handle, _dev(k, "k"), _dev(v, "v"), _dtype_code(k), k.shape[0],
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(q, "q"), _dtype_code(q), _dev(cache, "cache"),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(tail_k, "tail_k"), _dev(tail_v, "tail_v"), _dev(tail_lens, "tail_lens", torch.int32), float(scale),
        q.shape[0], _dev(out, "out"), _dtype_code(out) | (TQ_OUT_ROTATED if rotated else 0), _stream_ptr(stream)),
        "tq_store_decode_attention")


def tq_decode_attention_noalloc(handle, q, cache, block_table, seq_lens, out, tail_k=None, tail_v=None,
                                tail_lens=None, scale=0.0, stream=None):
    """tq_decode_attention with its scratch in the library's static device
    array instead of the handle's workspace (allocates nothing)."""
    import torch

    if tail_k is not None:
        _dev(tail_k, "tail_k", torch.bfloat16)
        _dev(tail_v, "tail_v", torch.bfloat16)
    _check(load_library().tq_decode_attention_noalloc(
        handle, _dev(q, "q"), _dtype_code(q), _dev(cache, "cache"), _dev(block_table, "block_table", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), _dev(tail_k, "tail_k"), _dev(tail_v, "tail_v"),
        _dev(tail_lens, "tail_lens", torch.int32), float(scale), q.shape[0], _dev(out, "out"), _dtype_code(out),
        _stream_ptr(stream)), "tq_decode_attention_noalloc")


def tq_extend_attention(handle, q, cache, block_table, prefix_lens, cu_q, new_k, new_v, out, scale=0.0, stream=None,
                        rotated=False):
    """q [T, H_q, d] (f32/bf16); block_table int32 [B, max_blocks_per_seq];
    prefix_lens int32 [B]; cu_q int32 [B+1]; new_k, new_v bf16 [T, H_kv, d];
    out [T, H_q, d] (f32/bf16)."""
    import torch

    T = q.shape[0]
    if new_k.shape != new_v.shape or new_k.shape[0] != T or out.shape != q.shape:
        raise ValueError("q, new_k, new_v and out must share the token count (out shaped like q)")
    if cu_q.shape[0] != prefix_lens.shape[0] + 1 or block_table.shape[0] < prefix_lens.shape[0]:
        raise ValueError("cu_q must have batch+1 entries and block_table at least batch rows")
    _check(load_library().tq_extend_attention(
        handle, _dev(q, "q"), _dtype_code(q), _dev(cache, "cache"), _dev(block_table, "block_table", torch.int32),
        _dev(prefix_lens, "prefix_lens", torch.int32), _dev(cu_q, "cu_q", torch.int32),
        _dev(new_k, "new_k", torch.bfloat16), _dev(new_v, "new_v", torch.bfloat16), float(scale),
        prefix_lens.shape[0], q.shape[0], _dev(out, "out"), _dtype_code(out) | (TQ_OUT_ROTATED if rotated else 0),
        _stream_ptr(stream)), "tq_extend_attention")


def tq_set_profile_events(handle, kernel, start=None, stop=None):
    """Record torch.cuda.Event pairs around the store (kernel=0) or decode
    split-KV (kernel=1) launch of later calls; None switches it off."""
    ev = lambda e: _P(e.cuda_event) if e is not None else _P()  # noqa: E731
    _check(load_library().tq_set_profile_events(handle, kernel, ev(start), ev(stop)), "tq_set_profile_events")


def tq_check_wait_timeout(err_word, limit_us, stream=None):
    """Make the decode kernels' bounded mbarrier wait run out (nothing ever
    completes the phase) with a limit of limit_us microseconds; the kernel ORs
    TQ_DEVERR_TIMEOUT into err_word (a CUDA uint32/int32 tensor of one
    element) and returns."""
    if err_word.numel() < 1 or err_word.element_size() != 4:
        raise ValueError("err_word must hold one 4-byte element")
    _check(load_library().tq_check_wait_timeout(_dev(err_word, "err_word"), int(limit_us), _stream_ptr(stream)),
           "tq_check_wait_timeout")


def tq_get_device_error(handle, stream=None):
    flags = ctypes.c_uint32()
    _check(load_library().tq_get_device_error(handle, ctypes.byref(flags), _stream_ptr(stream)),
           "tq_get_device_error")
    return flags.value


class TQCache:
    """Owns the device buffers of one cache configuration (torch uint8 tensors)
    and the library handle."""

    def __init__(self, device="cuda", **cfg_kwargs):
        import torch

        self.cfg = tq_cache_config(**cfg_kwargs)
        self.sizes = tq_cache_sizes(self.cfg)
        self.device = torch.device(device)
        self.params = torch.empty(self.sizes["params_bytes"], dtype=torch.uint8, device=self.device)
        self.workspace = torch.empty(self.sizes["workspace_bytes"], dtype=torch.uint8, device=self.device)
        self.cache = torch.zeros(self.sizes["cache_bytes"], dtype=torch.uint8, device=self.device)
        self.handle = tq_cache_create(self.cfg, self.params, self.workspace)

    @property
    def page_bytes(self):
        return self.sizes["page_bytes"]

    def pages(self):
        """The cache as [num_blocks, H_kv, page_bytes]."""
        return self.cache.view(self.cfg.num_blocks, self.cfg.num_kv_heads, self.page_bytes)

    def store(self, k, v, slot_mapping, stream=None):
        tq_store(self.handle, k, v, slot_mapping, self.cache, stream)

    def decode(self, q, block_table, seq_lens, out=None, tail_k=None, tail_v=None, tail_lens=None, scale=0.0,
               stream=None, out_dtype=None, rotated=False):
        import torch

        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype or torch.float32, device=q.device)
        tq_decode_attention(self.handle, q, self.cache, block_table, seq_lens, out, tail_k, tail_v, tail_lens,
                            scale, stream, rotated)
        return out

    def store_decode(self, k, v, slot_mapping, q, block_table, seq_lens, out=None, tail_k=None, tail_v=None,
                     tail_lens=None, scale=0.0, stream=None, out_dtype=None, rotated=False):
        import torch

        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype or torch.float32, device=q.device)
        tq_store_decode_attention(self.handle, k, v, slot_mapping, q, self.cache, block_table, seq_lens, out,
                                  tail_k, tail_v, tail_lens, scale, stream, rotated)
        return out

    def extend(self, q, block_table, prefix_lens, cu_q, new_k, new_v, out=None, scale=0.0, stream=None,
               out_dtype=None, rotated=False):
        import torch

        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype or torch.float32, device=q.device)
        tq_extend_attention(self.handle, q, self.cache, block_table, prefix_lens, cu_q, new_k, new_v, out, scale,
                            stream, rotated)
        return out

    def device_error(self, stream=None):
        return tq_get_device_error(self.handle, stream)

    def export_params(self):
        return tq_cache_export_params(self.handle, self.cfg)

    def close(self):
        if self.handle:
            tq_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
