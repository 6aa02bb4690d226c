"""Python binding of libspecverify (argument marshalling only).

The functions carry the C ABI's names and take torch CUDA tensors; every
step of the verify path runs in the library's CUDA kernels.  If the
library has not been built this module raises on first use: there is no
CPU fallback.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

(SV_OK, SV_EINVAL, SV_EBADTEMP, SV_EBADTOKEN, SV_EBADLOGIT, SV_ECUDA, SV_ESCRATCH, SV_EBADTREE,
 SV_EBADKV, SV_ETIMEOUT) = range(10)
SV_ERRBIT_TEMP, SV_ERRBIT_TOKEN, SV_ERRBIT_LOGIT, SV_ERRBIT_TREE, SV_ERRBIT_KV, SV_ERRBIT_WAIT = 1, 2, 4, 8, 16, 32
SV_KV_SCRATCH, SV_KV_INPLACE = 0, 1
SV_NORM_NONE, SV_NORM_LAYER, SV_NORM_RMS = 0, 1, 2
SV_TREE_SAMPLED, SV_TREE_TOPK = 0, 1
SV_F32, SV_BF16 = 0, 1
SV_NUM_KERNELS = 2
SV_MAX_N = 255
SV_NOALLOC_SCRATCH_BYTES = 1 << 20
KERNEL_NAMES = ("k0", "k1")  # profiling slots: row statistics, then walk and draws

_DTYPE_CODE = {torch.float32: SV_F32, torch.bfloat16: SV_BF16}

#: every symbol include/spec_verify.h declares
EXPORTS = (
    "spec_verify_init", "spec_verify", "spec_verify_get_error", "spec_verify_debug_stats",
    "spec_verify_profile", "spec_verify_profile_read", "spec_verify_launches_per_call",
    "spec_verify_debug_philox", "spec_verify_debug_read_stream", "spec_verify_destroy", "spec_verify_strerror",
    "spec_verify_noalloc", "spec_verify_tree", "spec_verify_tree_lazy", "spec_verify_kv_commit",
    "spec_verify_lazy",
    "spec_verify_fc_norm", "spec_verify_debug_seek_calls", "spec_verify_debug_skip_row_stats",
    "spec_verify_debug_late_cta",
)

_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


def load():
    """Load the shared library (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libspecverify.so is not built ({LIB_PATH}); run "
            "`python -m speculative_decoding_verification_73_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    c_int, c_void, c_u64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64
    lib.spec_verify_init.argtypes = [ctypes.POINTER(c_void), c_int, c_int, c_int, c_int, c_void]
    lib.spec_verify.argtypes = [c_void, c_int, c_int, c_int, c_void, c_void, c_void, c_void,
                                c_u64, c_void, c_void, c_void]
    lib.spec_verify_get_error.argtypes = [c_void, ctypes.POINTER(ctypes.c_uint32)]
    lib.spec_verify_debug_stats.argtypes = [c_void, c_int, c_int, c_void, c_void]
    lib.spec_verify_profile.argtypes = [c_void, c_int]
    lib.spec_verify_profile_read.argtypes = [c_void, ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(c_int)]
    lib.spec_verify_launches_per_call.argtypes = []
    lib.spec_verify_debug_philox.argtypes = [c_u64, c_void, c_void, c_int, c_void]
    lib.spec_verify_debug_read_stream.argtypes = [c_void, ctypes.c_size_t, c_void, c_void]
    lib.spec_verify_debug_seek_calls.argtypes = [c_void, ctypes.c_uint32]
    lib.spec_verify_debug_skip_row_stats.argtypes = [c_void, c_int]
    lib.spec_verify_debug_late_cta.argtypes = [c_void, c_int]
    lib.spec_verify_destroy.argtypes = [c_void]
    lib.spec_verify_lazy.argtypes = list(lib.spec_verify.argtypes)
    lib.spec_verify_fc_norm.argtypes = [c_void, c_int, c_int, c_int, c_int, ctypes.c_float, c_void,
                                        c_void, c_void, c_void, c_void, c_void, c_void, c_void, c_void]
    lib.spec_verify_kv_commit.argtypes = [c_void, c_int, c_int, c_int, c_int, c_int, ctypes.c_size_t,
                                          c_void, c_void, c_void, c_void, c_void, c_int]
    lib.spec_verify_tree.argtypes = [c_void, c_int, c_int, c_int, c_int, c_void, c_void, c_void,
                                     c_void, c_void, c_u64, c_void, c_void, c_void, c_void]
    lib.spec_verify_tree_lazy.argtypes = list(lib.spec_verify_tree.argtypes)
    lib.spec_verify_noalloc.argtypes = [c_int, c_int, c_int, c_int, c_void, c_void, c_void, c_void,
                                        c_u64, c_void, c_void, c_void, c_void]
    lib.spec_verify_strerror.argtypes = [c_int]
    lib.spec_verify_strerror.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name != "spec_verify_strerror":
            getattr(lib, name).restype = c_int
    _lib = lib
    return lib


def strerror(code):
    return load().spec_verify_strerror(int(code)).decode()


def _check(code, where):
    if code != SV_OK:
        raise SpecVerifyError(code, where)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def spec_verify_init(max_B, max_N, max_V, dtype, stream=None):
    """Create a context; returns its opaque handle (a ctypes void pointer)."""
    code = _DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    ctx = ctypes.c_void_p()
    _check(load().spec_verify_init(ctypes.byref(ctx), int(max_B), int(max_N), int(max_V), code,
                                   _stream_handle(stream)), "spec_verify_init")
    return ctx


def _require(t, name, shape, dtypes):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if tuple(t.shape) != tuple(shape) and t.numel() != int(np_prod(shape)):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}")


def np_prod(shape):
    n = 1
    for s in shape:
        n *= int(s)
    return n


def spec_verify(ctx, target_logits, draft_logits, draft_tokens, temperature, seed,
                out_tokens, out_accept_len, out_kv_len):
    """Enqueue one verify step; shapes are taken from ``target_logits``.
    Tensors must be contiguous CUDA tensors in the documented layouts."""
    B, n1, V = target_logits.shape
    logit_dt = (torch.float32, torch.bfloat16)
    _require(target_logits, "target_logits", (B, n1, V), logit_dt)
    if n1 > 1:
        _require(draft_logits, "draft_logits", (B, n1 - 1, V), (target_logits.dtype,))
        _require(draft_tokens, "draft_tokens", (B, n1 - 1), (torch.int32,))
    _require(temperature, "temperature", (B,), (torch.float32,))
    _require(out_tokens, "out_tokens", (B, n1), (torch.int32,))
    _require(out_accept_len, "out_accept_len", (B,), (torch.int32,))
    _require(out_kv_len, "out_kv_len", (B,), (torch.int32,))
    _check(load().spec_verify(ctx, int(B), int(n1 - 1), int(V), _ptr(target_logits),
                              _ptr(draft_logits), _ptr(draft_tokens), _ptr(temperature),
                              ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), _ptr(out_tokens),
                              _ptr(out_accept_len), _ptr(out_kv_len)), "spec_verify")


def spec_verify_noalloc(target_logits, draft_logits, draft_tokens, temperature, seed,
                        out_tokens, out_accept_len, out_kv_len, stream=None):
    """The verify step through the library's static scratch array: no context
    and no device allocation by the library (the caller owns every tensor).
    Enqueued on ``stream`` (default: torch's current stream).  Raises
    SpecVerifyError with code SV_ESCRATCH when the problem's working memory
    exceeds SV_NOALLOC_SCRATCH_BYTES."""
    B, n1, V = target_logits.shape
    logit_dt = (torch.float32, torch.bfloat16)
    _require(target_logits, "target_logits", (B, n1, V), logit_dt)
    if n1 > 1:
        _require(draft_logits, "draft_logits", (B, n1 - 1, V), (target_logits.dtype,))
        _require(draft_tokens, "draft_tokens", (B, n1 - 1), (torch.int32,))
    _require(temperature, "temperature", (B,), (torch.float32,))
    _require(out_tokens, "out_tokens", (B, n1), (torch.int32,))
    _require(out_accept_len, "out_accept_len", (B,), (torch.int32,))
    _require(out_kv_len, "out_kv_len", (B,), (torch.int32,))
    _check(load().spec_verify_noalloc(int(B), int(n1 - 1), int(V), _DTYPE_CODE[target_logits.dtype],
                                      _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens),
                                      _ptr(temperature),
                                      ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF),
                                      _ptr(out_tokens), _ptr(out_accept_len), _ptr(out_kv_len),
                                      _stream_handle(stream)), "spec_verify_noalloc")


def spec_verify_tree(ctx, mode, target_logits, draft_logits, parents, draft_tokens, temperature,
                     seed, out_tokens, out_path, out_accept_len, out_kv_len, lazy=False):
    """Enqueue one tree verify step; B, M, V are taken from ``target_logits``
    [B, M+1, V].  ``draft_logits`` [B, M+1, V] may be None in TOPK mode.
    ``lazy`` calls spec_verify_tree_lazy (rows read only where the walk goes)."""
    B, m1, V = target_logits.shape
    M = m1 - 1
    logit_dt = (torch.float32, torch.bfloat16)
    _require(target_logits, "target_logits", (B, m1, V), logit_dt)
    if mode == SV_TREE_SAMPLED and M > 0:
        _require(draft_logits, "draft_logits", (B, m1, V), (target_logits.dtype,))
    if M > 0:
        _require(parents, "parents", (B, M), (torch.int32,))
        _require(draft_tokens, "draft_tokens", (B, M), (torch.int32,))
        _require(out_path, "out_path", (B, M), (torch.int32,))
    _require(temperature, "temperature", (B,), (torch.float32,))
    _require(out_tokens, "out_tokens", (B, m1), (torch.int32,))
    _require(out_accept_len, "out_accept_len", (B,), (torch.int32,))
    _require(out_kv_len, "out_kv_len", (B,), (torch.int32,))
    name = "spec_verify_tree_lazy" if lazy else "spec_verify_tree"
    _check(getattr(load(), name)(ctx, int(B), int(M), int(V), int(mode), _ptr(target_logits),
                                 _ptr(draft_logits), _ptr(parents), _ptr(draft_tokens),
                                 _ptr(temperature), ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF),
                                 _ptr(out_tokens), _ptr(out_path), _ptr(out_accept_len),
                                 _ptr(out_kv_len)), name)


def spec_verify_kv_commit(ctx, mode, cache, seq_len, kv_len, scratch=None, path=None):
    """Commit the kept window entries.  cache [L, B, S, E] and scratch
    [L, B, W, E] are uint8 CUDA tensors (E bytes per layer and position);
    seq_len [B] int32 is advanced in place; path [B, P] int32 (a tree's
    out_path) or None for a chain."""
    if cache.dim() != 4 or cache.dtype != torch.uint8:
        raise ValueError("cache must be a uint8 tensor [L, B, S, E]")
    L, B, S, E = cache.shape
    _require(cache, "cache", (L, B, S, E), (torch.uint8,))
    _require(seq_len, "seq_len", (B,), (torch.int32,))
    _require(kv_len, "kv_len", (B,), (torch.int32,))
    W = 0
    if mode == SV_KV_SCRATCH:
        _require(scratch, "scratch", scratch.shape, (torch.uint8,))
        if scratch.dim() != 4 or tuple(scratch.shape[:2]) != (L, B) or scratch.shape[3] != E:
            raise ValueError("scratch must be [L, B, W, E] like the cache")
        W = scratch.shape[2]
    stride = 0
    if path is not None:
        _require(path, "path", path.shape, (torch.int32,))
        stride = path.shape[1]
    _check(load().spec_verify_kv_commit(ctx, int(mode), int(L), int(B), int(S), int(W), int(E),
                                        _ptr(scratch), _ptr(cache), _ptr(seq_len), _ptr(kv_len),
                                        _ptr(path), int(stride)), "spec_verify_kv_commit")


def spec_verify_lazy(ctx, target_logits, draft_logits, draft_tokens, temperature, seed,
                     out_tokens, out_accept_len, out_kv_len):
    """spec_verify that reads each request's rows only as far as its walk
    goes (same arguments and outputs)."""
    B, n1, V = target_logits.shape
    logit_dt = (torch.float32, torch.bfloat16)
    _require(target_logits, "target_logits", (B, n1, V), logit_dt)
    if n1 > 1:
        _require(draft_logits, "draft_logits", (B, n1 - 1, V), (target_logits.dtype,))
        _require(draft_tokens, "draft_tokens", (B, n1 - 1), (torch.int32,))
    _require(temperature, "temperature", (B,), (torch.float32,))
    _require(out_tokens, "out_tokens", (B, n1), (torch.int32,))
    _require(out_accept_len, "out_accept_len", (B,), (torch.int32,))
    _require(out_kv_len, "out_kv_len", (B,), (torch.int32,))
    _check(load().spec_verify_lazy(ctx, int(B), int(n1 - 1), int(V), _ptr(target_logits),
                                   _ptr(draft_logits), _ptr(draft_tokens), _ptr(temperature),
                                   ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), _ptr(out_tokens),
                                   _ptr(out_accept_len), _ptr(out_kv_len)), "spec_verify_lazy")


def spec_verify_fc_norm(ctx, norm, h_early, h_mid, h_late, weight, gamma=None, beta=None,
                        bias=None, eps=1e-5, out=None, xbuf=None):
    """out [T, d_out] bf16 = [norm(h_early); norm(h_mid); norm(h_late)] . W^T
    + bias.  h_*: [T, d] bf16 CUDA tensors; weight [d_out, 3d] bf16; gamma /
    beta [3, d] and bias [d_out] float32.  Returns out."""
    T, d = h_early.shape
    d_out = weight.shape[0]
    for name, h in (("h_early", h_early), ("h_mid", h_mid), ("h_late", h_late)):
        _require(h, name, (T, d), (torch.bfloat16,))
    _require(weight, "weight", (d_out, 3 * d), (torch.bfloat16,))
    if gamma is not None:
        _require(gamma, "gamma", (3, d), (torch.float32,))
    if beta is not None:
        _require(beta, "beta", (3, d), (torch.float32,))
    if bias is not None:
        _require(bias, "bias", (d_out,), (torch.float32,))
    if out is None:
        out = torch.empty(T, d_out, dtype=torch.bfloat16, device=h_early.device)
    _require(out, "out", (T, d_out), (torch.bfloat16,))
    if xbuf is None:
        xbuf = torch.empty(T, 3 * d, dtype=torch.bfloat16, device=h_early.device)
    _require(xbuf, "xbuf", (T, 3 * d), (torch.bfloat16,))
    _check(load().spec_verify_fc_norm(ctx, int(T), int(d), int(d_out), int(norm), float(eps),
                                      _ptr(h_early), _ptr(h_mid), _ptr(h_late), _ptr(gamma), _ptr(beta),
                                      _ptr(weight), _ptr(bias), _ptr(out), _ptr(xbuf)),
           "spec_verify_fc_norm")
    return out


def spec_verify_get_error(ctx):
    """(code, bits) of the device-detected input errors since the last read."""
    bits = ctypes.c_uint32(0)
    code = load().spec_verify_get_error(ctx, ctypes.byref(bits))
    if code in (SV_ECUDA, SV_EINVAL):
        raise SpecVerifyError(code, "spec_verify_get_error")
    return code, int(bits.value)


def spec_verify_debug_stats(ctx, B, N, device=None):
    """(accept_prob [B, N], log_z [B, 2N+1]) of the last call, as CUDA tensors."""
    acc = torch.empty(B, N, dtype=torch.float32, device=device or "cuda")
    lz = torch.empty(B, 2 * N + 1, dtype=torch.float32, device=device or "cuda")
    _check(load().spec_verify_debug_stats(ctx, int(B), int(N), _ptr(acc), _ptr(lz)),
           "spec_verify_debug_stats")
    return acc, lz


def spec_verify_profile(ctx, every):
    """Record kernel events on every ``every``-th call (True = 1 = all calls;
    0 or False = off)."""
    _check(load().spec_verify_profile(ctx, int(every)), "spec_verify_profile")


def spec_verify_profile_read(ctx):
    """({kernel name: summed ms}, recorded calls) since the last read."""
    ms = (ctypes.c_double * SV_NUM_KERNELS)()
    calls = ctypes.c_int(0)
    _check(load().spec_verify_profile_read(ctx, ms, ctypes.byref(calls)), "spec_verify_profile_read")
    return dict(zip(KERNEL_NAMES, list(ms))), int(calls.value)


def spec_verify_launches_per_call():
    return int(load().spec_verify_launches_per_call())


def spec_verify_debug_philox(seed, counters, stream=None):
    """Philox4x32-10 words for counters [n, 3] (uint32 values in an int32 or
    int64 CUDA tensor); returns [n, 4] int64 tensor of the 32-bit words."""
    ctr = counters.to(torch.int32).contiguous()
    n = ctr.shape[0]
    out = torch.empty(n, 4, dtype=torch.int32, device=ctr.device)
    _check(load().spec_verify_debug_philox(ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF),
                                           _ptr(ctr), _ptr(out), int(n), _stream_handle(stream)),
           "spec_verify_debug_philox")
    return out.to(torch.int64) & 0xFFFFFFFF


def spec_verify_debug_read_stream(buf, out=None, stream=None):
    """Read the CUDA tensor buf (contiguous, 16-byte aligned, a multiple of
    16 bytes) once on the device, adding the sum of its 64-bit words modulo
    2^64 to the one-element int64 CUDA tensor out (a new zeroed one when
    None); returns out."""
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    nbytes = buf.numel() * buf.element_size()
    if out is None:
        out = torch.zeros(1, dtype=torch.int64, device=buf.device)
    _check(load().spec_verify_debug_read_stream(_ptr(buf), int(nbytes), _ptr(out), _stream_handle(stream)),
           "spec_verify_debug_read_stream")
    return out


def spec_verify_destroy(ctx):
    _check(load().spec_verify_destroy(ctx), "spec_verify_destroy")


class SpecVerify:
    """A context plus preallocated outputs: ``sv(target, draft, tokens, T, seed)``
    returns (out_tokens, out_accept_len, out_kv_len) as CUDA tensors."""

    def __init__(self, max_B, max_N, max_V, dtype, stream=None, device=None):
        self.max_B, self.max_N, self.max_V, self.dtype = max_B, max_N, max_V, dtype
        self.device = torch.device(device or "cuda")
        self.stream = stream
        self.ctx = spec_verify_init(max_B, max_N, max_V, dtype, stream)
        self.out_tokens = torch.empty(max_B * (max_N + 1), dtype=torch.int32, device=self.device)
        self.out_accept = torch.empty(max_B, dtype=torch.int32, device=self.device)
        self.out_kv = torch.empty(max_B, dtype=torch.int32, device=self.device)
        self.out_path = torch.empty(max_B * max(max_N, 1), dtype=torch.int32, device=self.device)

    def __call__(self, target, draft, tokens, temperature, seed):
        B, n1, _ = target.shape
        toks = self.out_tokens[: B * n1].view(B, n1)
        acc, kv = self.out_accept[:B], self.out_kv[:B]
        spec_verify(self.ctx, target, draft, tokens, temperature, seed, toks, acc, kv)
        return toks, acc, kv

    def lazy(self, target, draft, tokens, temperature, seed):
        """spec_verify_lazy into this context's output buffers."""
        B, n1, _ = target.shape
        toks = self.out_tokens[: B * n1].view(B, n1)
        acc, kv = self.out_accept[:B], self.out_kv[:B]
        spec_verify_lazy(self.ctx, target, draft, tokens, temperature, seed, toks, acc, kv)
        return toks, acc, kv

    def tree(self, target, draft, parents, tokens, temperature, seed, mode=SV_TREE_SAMPLED, lazy=False):
        """Tree verify (``lazy``: spec_verify_tree_lazy); returns (out_tokens
        [B, M+1], out_path [B, M], out_accept_len [B], out_kv_len [B]) as CUDA
        tensors."""
        B, m1, _ = target.shape
        toks = self.out_tokens[: B * m1].view(B, m1)
        path = self.out_path[: B * (m1 - 1)].view(B, m1 - 1)
        acc, kv = self.out_accept[:B], self.out_kv[:B]
        spec_verify_tree(self.ctx, mode, target, draft, parents, tokens, temperature, seed,
                         toks, path, acc, kv, lazy=lazy)
        return toks, path, acc, kv

    def get_error(self):
        return spec_verify_get_error(self.ctx)

    def debug_skip_row_stats(self, on):
        """Test hook: walk kernels alone (see spec_verify_debug_skip_row_stats)."""
        _check(load().spec_verify_debug_skip_row_stats(self.ctx, 1 if on else 0),
               "spec_verify_debug_skip_row_stats")

    def debug_late_cta(self, cta):
        """Test hook: sampler CTA `cta` of every request acts as if its wait
        ran out; -1 = off (see spec_verify_debug_late_cta)."""
        _check(load().spec_verify_debug_late_cta(self.ctx, int(cta)), "spec_verify_debug_late_cta")

    def debug_seek_calls(self, calls):
        """Test hook: set the context's call count (see spec_verify_debug_seek_calls)."""
        _check(load().spec_verify_debug_seek_calls(self.ctx, int(calls) & 0xFFFFFFFF),
               "spec_verify_debug_seek_calls")

    def debug_stats(self, B, N):
        return spec_verify_debug_stats(self.ctx, B, N, self.device)

    def close(self):
        if self.ctx is not None:
            spec_verify_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
