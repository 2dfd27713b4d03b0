"""GB300 speculative-decoding verification step -- Python binding.

A thin ctypes layer over the C ABI in ``include/specverify.h``: it marshals
arguments and raises on error codes.  Every step of the path runs in the
CUDA library (``_lib/libspecverify.so``, built by ``build()``); there is no
CPU fallback, and using the binding without the built library raises.
Device memory (weights, logits) is passed as torch CUDA tensors, read by
pointer.
"""
import ctypes
import os

from ._build import LIB, build

__all__ = ["build", "lib", "SpecError", "SpecDecoder", "accept_rows", "sample_rows",
           "SPEC_DTYPE_F32", "SPEC_DTYPE_BF16", "SPEC_OPT_NO_GRAPH", "SPEC_OPT_TIMING",
           "SPEC_FLAG_RESID_ZERO", "SPEC_FLAG_ALL_ACCEPTED"]

SPEC_OK = 0
ERRORS = {-1: "SPEC_E_ARG", -2: "SPEC_E_VOCAB", -3: "SPEC_E_SHAPE", -4: "SPEC_E_CAPACITY",
          -5: "SPEC_E_CUDA", -6: "SPEC_E_OOM", -7: "SPEC_E_TIMEOUT", -8: "SPEC_E_STATE"}
SPEC_DTYPE_F32 = 0
SPEC_DTYPE_BF16 = 1
SPEC_DTYPE_Q4 = 2
_DTYPES = {"f32": SPEC_DTYPE_F32, "bf16": SPEC_DTYPE_BF16, "q4": SPEC_DTYPE_Q4}
SPEC_MAX_BATCH = 64
SPEC_FLAG_RESID_ZERO = 0x1
SPEC_FLAG_ALL_ACCEPTED = 0x2
SPEC_OPT_NO_GRAPH = 0x1
SPEC_OPT_TIMING = 0x2
SPEC_OPT_PDL = 0x4
SPEC_OPT_NO_PERSIST = 0x8
SPEC_OPT_PHASE_TIMES = 0x10
SPEC_FAULT_CLEAR = 0
SPEC_FAULT_ALLOC = 1
SPEC_FAULT_WAIT_TIMEOUT = 2

_LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LAYER_FIELDS]


class ModelDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn_dim", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("dtype", ctypes.c_int), ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerWeights))]


class Opts(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("max_ctx", ctypes.c_int), ("temperature", ctypes.c_float),
                ("seed", ctypes.c_uint64), ("draft_mix_lambda", ctypes.c_float),
                ("cuda_stream", ctypes.c_void_p), ("flags", ctypes.c_int), ("draft_lookup", ctypes.c_int),
                ("draft_heads", ctypes.c_void_p)]


class Stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("ar_steps", ctypes.c_int64),
                ("tokens_emitted", ctypes.c_int64), ("drafts_accepted", ctypes.c_int64),
                ("accept_hist", ctypes.c_int64 * 17), ("context_len", ctypes.c_int32),
                ("kernels_per_step", ctypes.c_int32), ("kernels_per_ar_step", ctypes.c_int32),
                ("gemm_launches_per_verify", ctypes.c_int32),
                ("verify_weight_bytes", ctypes.c_double), ("draft_weight_bytes", ctypes.c_double),
                ("kv_bytes_per_token_target", ctypes.c_double),
                ("kv_bytes_per_token_draft", ctypes.c_double),
                ("timed_gemm_ms", ctypes.c_double), ("timed_gemm_bytes", ctypes.c_double),
                ("timed_gemm_launches", ctypes.c_int64)]

    def as_dict(self):
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["accept_hist"] = list(self.accept_hist)
        return d


class Profile(ctypes.Structure):
    _fields_ = [("draft_loop_ms", ctypes.c_double), ("verify_ms", ctypes.c_double),
                ("ar_ms", ctypes.c_double), ("iters", ctypes.c_int32),
                ("kernels_draft_loop", ctypes.c_int32), ("kernels_verify", ctypes.c_int32),
                ("kernels_ar", ctypes.c_int32), ("verify_forward_ms", ctypes.c_double),
                ("kernels_verify_forward", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_I32P = ctypes.POINTER(ctypes.c_int32)
_U32P = ctypes.POINTER(ctypes.c_uint32)
_F32P = ctypes.POINTER(ctypes.c_float)
_VP = ctypes.c_void_p

# name -> (restype, argtypes); every function declared in include/specverify.h
SIGNATURES = {
    "spec_init": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(ModelDesc), ctypes.c_int,
                                 ctypes.POINTER(Opts), ctypes.POINTER(_VP)]),
    "spec_free": (None, [_VP]),
    "spec_last_error": (ctypes.c_char_p, [_VP]),
    "spec_prefill": (ctypes.c_int, [_VP, _I32P, ctypes.c_int]),
    "spec_prefill_synthetic": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_uint64]),
    "spec_seq_context": (ctypes.c_int, [_VP, ctypes.c_int, _I32P, _I32P]),
    "spec_step": (ctypes.c_int, [_VP, _I32P, _I32P, _U32P]),
    "spec_generate": (ctypes.c_int, [_VP, ctypes.c_int, _I32P, _I32P]),
    "spec_ar_step": (ctypes.c_int, [_VP, _I32P]),
    "spec_get_stats": (ctypes.c_int, [_VP, ctypes.POINTER(Stats)]),
    "spec_last_step_debug": (ctypes.c_int, [_VP, _F32P, _F32P, _I32P, _I32P, _I32P]),
    "spec_model_forward": (ctypes.c_int, [_VP, ctypes.c_int, _I32P, ctypes.c_int, ctypes.c_int, _VP]),
    "spec_accept_rows": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, ctypes.c_int64, _VP, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_uint64,
                                        ctypes.c_uint64, _VP, _VP, _VP, _VP]),
    "spec_accept_rows_noalloc": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, ctypes.c_int64, _VP,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64,
                                                _VP, _VP, _VP, _VP]),
    "spec_sample_rows": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_int, _VP, _VP]),
    "spec_profile": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(Profile)]),
    "spec_phase_times": (ctypes.c_int, [_VP, ctypes.c_int, _VP, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int)]),
    "spec_version": (ctypes.c_char_p, []),
    "spec_inject_fault": (ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int]),
    "spec_phase_list": (ctypes.c_int, [_VP, ctypes.c_int, _VP, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    "spec_device_bytes_held": (ctypes.c_int64, []),
}

_lib = None


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run build() first; this package has no CPU fallback")
        handle = ctypes.CDLL(LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class SpecError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def _check(rc, ctx=None):
    if rc != SPEC_OK:
        msg = lib().spec_last_error(ctx).decode(errors="replace")
        raise SpecError(rc, msg)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def model_desc(shape, weights):
    """ModelDesc for a shape (attributes n_layers, d_model, n_heads, n_kv_heads,
    head_dim, ffn_dim, vocab, rope_theta, rms_eps, dtype 'f32'|'bf16'|'q4') and a
    weights dict {'embed', 'final_norm', 'lm_head', 'layers': [dict]} of CUDA
    tensors ('q4': every matrix one uint8 buffer of packed codes followed by
    group-major bf16 scales, see include/specverify.h).  Returns (desc, keepalive)."""
    layers = (LayerWeights * shape.n_layers)()
    for i, lw in enumerate(weights["layers"]):
        for n in _LAYER_FIELDS:
            setattr(layers[i], n, lw[n].data_ptr())
    d = ModelDesc(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                  shape.ffn_dim, shape.vocab, shape.rope_theta, shape.rms_eps, _DTYPES[shape.dtype],
                  weights["embed"].data_ptr(), weights["final_norm"].data_ptr(),
                  weights["lm_head"].data_ptr(), layers)
    return d, (layers, weights)


class SpecDecoder:
    """One target/draft pair with K drafts per step over `batch` sequences
    (batch > 1: bf16 models, every sequence advancing independently);
    lookup = n > 0 drafts by prompt lookup (n-gram suffix match up to n
    tokens) instead of running the draft model; heads = a device tensor
    [K, d_model, d_model] in the target's arithmetic dtype drafts with
    self-draft heads on the target (draft_shape / draft_w then None)."""

    def __init__(self, target_shape, target_w, draft_shape, draft_w, k, max_ctx,
                 temperature=0.0, seed=0, mix_lambda=0.0, stream=None, flags=0, batch=1, lookup=0,
                 heads=None):
        self.k = k
        self.batch = batch
        self.vocab = target_shape.vocab
        self._td, self._tk = model_desc(target_shape, target_w)
        self._heads = heads
        if draft_shape is None:
            self._dd, self._dk = None, None
        else:
            self._dd, self._dk = model_desc(draft_shape, draft_w)
        opts = Opts(batch, max_ctx, temperature, seed, mix_lambda,
                    ctypes.c_void_p(stream) if stream else ctypes.c_void_p(0), flags, lookup,
                    ctypes.c_void_p(heads.data_ptr() if heads is not None else 0))
        h = ctypes.c_void_p()
        rc = lib().spec_init(ctypes.byref(self._td), ctypes.byref(self._dd) if self._dd is not None else None, k,
                             ctypes.byref(opts), ctypes.byref(h))
        _check(rc)
        self.ctx = h

    def close(self):
        if getattr(self, "ctx", None):
            lib().spec_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens):
        """tokens: one prompt (batch 1) or `batch` prompts of one length."""
        rows = [list(tokens)] if self.batch == 1 and not hasattr(tokens[0], "__len__") else list(tokens)
        n = len(rows[0])
        flat = [int(t) for r in rows for t in r]
        arr = (ctypes.c_int32 * len(flat))(*flat)
        _check(lib().spec_prefill(self.ctx, arr, n), self.ctx)

    def prefill_synthetic(self, length, seed=0):
        """State of a prefill of `length` tokens with synthetic token ids and
        KV caches (benchmark workloads; the tokens carry no meaning)."""
        _check(lib().spec_prefill_synthetic(self.ctx, length, seed), self.ctx)

    def step(self):
        """Batch 1: (emitted tokens, flags).  Batch > 1: ([tokens of each
        sequence], [flags of each sequence])."""
        b = self.batch
        out = (ctypes.c_int32 * (b * (self.k + 1)))()
        cnt = (ctypes.c_int32 * b)()
        flags = (ctypes.c_uint32 * b)()
        _check(lib().spec_step(self.ctx, out, cnt, flags), self.ctx)
        rows = [list(out[i * (self.k + 1):i * (self.k + 1) + cnt[i]]) for i in range(b)]
        if b == 1:
            return rows[0], flags[0]
        return rows, list(flags)

    def seq_context(self, b):
        """Committed tokens of sequence b (the last is the pending token)."""
        import numpy as np
        n = ctypes.c_int32()
        _check(lib().spec_seq_context(self.ctx, b, None, ctypes.byref(n)), self.ctx)
        buf = np.zeros(max(1, n.value), dtype=np.int32)
        _check(lib().spec_seq_context(self.ctx, b, buf.ctypes.data_as(_I32P), ctypes.byref(n)), self.ctx)
        return buf[:n.value].copy()

    def generate(self, n_new):
        out = (ctypes.c_int32 * max(1, n_new))()
        got = ctypes.c_int32()
        _check(lib().spec_generate(self.ctx, n_new, out, ctypes.byref(got)), self.ctx)
        return list(out[:got.value])

    def ar_step(self):
        """Batch 1: the token; batch > 1: one token per sequence."""
        tok = (ctypes.c_int32 * self.batch)()
        _check(lib().spec_ar_step(self.ctx, tok), self.ctx)
        return tok[0] if self.batch == 1 else list(tok)

    def stats(self):
        s = Stats()
        _check(lib().spec_get_stats(self.ctx, ctypes.byref(s)), self.ctx)
        return s.as_dict()

    def profile(self, iters=20):
        """Graph-replayed phase times (ms): draft loop, verify pass, plain-decoding
        pass, and the verify pass's target forward alone."""
        pr = Profile()
        _check(lib().spec_profile(self.ctx, iters, ctypes.byref(pr)), self.ctx)
        return pr.as_dict()

    def phase_times(self, which):
        """Per-phase stamps of the last persistent run of forward `which`
        (0..K-1 draft passes, K verify, K+1 plain decoding): a list of dicts
        with kind, n, k, the earliest/latest arrival, the release, the latest
        end of X preparation and the latest end of streaming, in ns."""
        import numpy as np
        buf = np.zeros((1024, 8), dtype=np.int64)
        n = ctypes.c_int(0)
        _check(lib().spec_phase_times(self.ctx, which, buf.ctypes.data_as(_VP), 1024,
                                      ctypes.byref(n)), self.ctx)
        names = ("kind", "n", "k", "arrive_min_ns", "arrive_max_ns", "release_ns", "prep_max_ns",
                 "work_max_ns")
        return [dict(zip(names, (int(v) for v in row))) for row in buf[:n.value]]

    def last_step_debug(self, max_ctx):
        """(p_logits [K+1, V], q_logits [K, V], drafts [K], context tokens) as
        numpy; batch > 1: p [B, K+1, V], q [B, K, V], drafts [B, K] and
        sequence 0's context."""
        import numpy as np
        k, v, b = self.k, self.vocab, self.batch
        lead = () if b == 1 else (b,)
        p = np.zeros(lead + (k + 1, v), dtype=np.float32)
        q = np.zeros(lead + (k, v), dtype=np.float32)
        d = np.zeros(lead + (k,), dtype=np.int32)
        ctx = np.zeros(max_ctx, dtype=np.int32)
        n = ctypes.c_int32()
        _check(lib().spec_last_step_debug(self.ctx, p.ctypes.data_as(_F32P), q.ctypes.data_as(_F32P),
                                          d.ctypes.data_as(_I32P), ctx.ctypes.data_as(_I32P),
                                          ctypes.byref(n)), self.ctx)
        return p, q, d, ctx[:n.value].copy()

    def phase_list(self, which):
        """Phase geometry of persistent forward `which` (0..K-1 draft passes,
        K verify, K+1 plain decoding): a list of 8-tuples, see spec_phase_list."""
        import numpy as np
        buf = np.zeros((4096, 8), dtype=np.int64)
        n = ctypes.c_int(0)
        _check(lib().spec_phase_list(self.ctx, which, buf.ctypes.data_as(_VP), 4096, ctypes.byref(n)), self.ctx)
        return [tuple(int(v) for v in row) for row in buf[:n.value]]

    def inject_fault(self, kind, arg):
        """Test hook: arm (arg > 0) or disarm (0) a fault of this context
        (SPEC_FAULT_WAIT_TIMEOUT) -- see include/specverify.h."""
        _check(lib().spec_inject_fault(self.ctx, kind, arg), self.ctx)

    def model_forward(self, which, tokens, pos0, logits):
        """Forward of the target (0) or draft (1) over host token ids at
        positions pos0.. into logits (CUDA fp32 tensor [n, V])."""
        arr = (ctypes.c_int32 * len(tokens))(*[int(t) for t in tokens])
        _check(lib().spec_model_forward(self.ctx, which, arr, len(tokens), pos0, _ptr(logits)), self.ctx)


def inject_alloc_failure(n):
    """Test hook: the n-th device allocation of the next context creation fails."""
    _check(lib().spec_inject_fault(None, SPEC_FAULT_ALLOC, n))


def clear_faults():
    _check(lib().spec_inject_fault(None, SPEC_FAULT_CLEAR, 0))


def device_bytes_held():
    """Device bytes held by every live context of this process."""
    return int(lib().spec_device_bytes_held())


def accept_rows(p_logits, q_logits, drafts, temperature, seed, step_base=0, stream=None,
                p_row_stride=None, q_row_stride=None, rows=None):
    """Fused acceptance over independent verify rows (CUDA tensors):
    p_logits [R, K+1, V] fp32, q_logits [R, K, V] fp32, drafts [R, K] int32.
    Returns (tokens [R, K+1] int32, counts [R] int32, flags [R] int32)."""
    import torch
    K = q_logits.shape[-2]
    V = p_logits.shape[-1]
    R = rows if rows is not None else p_logits.shape[0]
    dev = p_logits.device
    tokens = torch.empty((R, K + 1), dtype=torch.int32, device=dev)
    counts = torch.empty(R, dtype=torch.int32, device=dev)
    flags = torch.empty(R, dtype=torch.int32, device=dev)
    ps = p_row_stride if p_row_stride is not None else (K + 1) * V
    qs = q_row_stride if q_row_stride is not None else K * V
    st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check(lib().spec_accept_rows(_ptr(p_logits), ps, _ptr(q_logits), qs, _ptr(drafts), R, K, V,
                                  float(temperature), int(seed), int(step_base), _ptr(tokens),
                                  _ptr(counts), _ptr(flags), ctypes.c_void_p(st)))
    return tokens, counts, flags


def accept_rows_noalloc(p_logits, q_logits, drafts, temperature, seed, step_base=0, stream=None):
    """accept_rows for callers that cannot allocate device memory: the library's
    scratch comes from a fixed 4 MiB array instead of an allocator (outputs are
    still torch tensors here; C callers pass their own buffers)."""
    import torch
    K = q_logits.shape[-2]
    V = p_logits.shape[-1]
    R = p_logits.shape[0]
    dev = p_logits.device
    tokens = torch.empty((R, K + 1), dtype=torch.int32, device=dev)
    counts = torch.empty(R, dtype=torch.int32, device=dev)
    flags = torch.empty(R, dtype=torch.int32, device=dev)
    st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check(lib().spec_accept_rows_noalloc(_ptr(p_logits), (K + 1) * V, _ptr(q_logits), K * V,
                                          _ptr(drafts), R, K, V, float(temperature), int(seed),
                                          int(step_base), _ptr(tokens), _ptr(counts), _ptr(flags),
                                          ctypes.c_void_p(st)))
    return tokens, counts, flags


def sample_rows(logits, temperature, seed, step_base=0, position=1, stream=None, row_stride=None,
                rows=None):
    """Inverse-CDF draw per row of logits [R, V] (CUDA fp32); returns int32 [R]."""
    import torch
    V = logits.shape[-1]
    R = rows if rows is not None else logits.shape[0]
    out = torch.empty(R, dtype=torch.int32, device=logits.device)
    st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rs = row_stride if row_stride is not None else V
    _check(lib().spec_sample_rows(_ptr(logits), rs, R, V, float(temperature), int(seed),
                                  int(step_base), int(position), _ptr(out), ctypes.c_void_p(st)))
    return out
