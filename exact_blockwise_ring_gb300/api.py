"""ctypes binding of libra.so (the C ABI in include/ra.h).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the library has
not been built, every call raises; there is no fallback path.
"""

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# RA_LIBRARY selects another build of the library (e.g. the checked build libra_checked.so)
LIB_PATH = os.environ.get("RA_LIBRARY") or os.path.join(_HERE, "libra.so")
HEADER_PATH = os.path.join(_HERE, "..", "include", "ra.h")

LAYOUTS = {"contiguous": 0, "striped": 1, "zigzag": 2}
STATUS = {0: "RA_OK", 1: "RA_ERR_INVALID_ARG", 2: "RA_ERR_UNSUPPORTED", 3: "RA_ERR_WORKSPACE",
          4: "RA_ERR_CUDA", 5: "RA_ERR_DEVICE_TIMEOUT", 6: "RA_ERR_CHECK"}
RA_BF16, RA_FP32 = 0, 1


class Params(ctypes.Structure):
    """Mirror of ra_params_t."""
    _fields_ = [("batch", ctypes.c_int), ("seq_len", ctypes.c_int64), ("heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("block", ctypes.c_int), ("P", ctypes.c_int),
                ("layout", ctypes.c_int), ("causal", ctypes.c_int),
                ("softmax_scale", ctypes.c_float), ("n_split", ctypes.c_int),
                ("kv_heads", ctypes.c_int)]


class BptParams(ctypes.Structure):
    """Mirror of ra_bpt_params_t."""
    _fields_ = [("attn", Params), ("d_ff", ctypes.c_int), ("block_rows", ctypes.c_int64),
                ("ln_eps", ctypes.c_float)]


BPT_WEIGHTS = ("wq", "wk", "wv", "wo", "w1", "w2", "bq", "bk", "bv", "bo", "b1", "b2",
               "ln1_g", "ln1_b", "ln2_g", "ln2_b")


class BptWeights(ctypes.Structure):
    """Mirror of ra_bpt_weights_t (device pointers)."""
    _fields_ = [(n, ctypes.c_void_p) for n in BPT_WEIGHTS]


class BptGrads(ctypes.Structure):
    """Mirror of ra_bpt_grads_t (device pointers)."""
    _fields_ = [("dx", ctypes.c_void_p)] + [(n, ctypes.c_void_p) for n in BPT_WEIGHTS]


EPILOGUES = {"bias": 0, "bias_gelu": 1, "bias_residual": 2}


class RaError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__("%s: %s" % (STATUS.get(status, status), message))


_lib = None
_lib_lock = threading.Lock()

_P = ctypes.c_void_p
_SIGS = {
    "ra_fwd_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Params)]),
    "ra_bwd_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Params)]),
    "ra_fwd": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P, ctypes.c_int, _P, _P, _P,
                              ctypes.c_size_t, _P]),
    "ra_bwd": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P, ctypes.c_int, _P, _P, _P,
                              _P, _P, _P, ctypes.c_size_t, _P]),
    "ra_bwd_preprocess": (ctypes.c_int, [ctypes.POINTER(Params), _P, ctypes.c_int, _P, _P, _P,
                                         ctypes.c_size_t, _P]),
    "ra_bwd_main": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _P, _P,
                                   ctypes.c_size_t, _P]),
    "ra_bwd_finalize": (ctypes.c_int, [ctypes.POINTER(Params), _P, _P, ctypes.c_size_t, _P]),
    "ra_merge": (ctypes.c_int, [ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                ctypes.c_int, _P, ctypes.c_int, _P, _P]),
    "ra_shard_work_model": (ctypes.c_int, [ctypes.POINTER(Params),
                                           ctypes.POINTER(ctypes.c_ulonglong)]),
    "ra_check_error": (ctypes.c_int, [_P, _P]),
    "ra_selftest_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint, _P]),
    "ra_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ra_linear": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P,
                                 ctypes.c_int, _P, _P, ctypes.c_size_t, _P]),
    "ra_layernorm": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, _P, _P, _P, ctypes.c_float, _P,
                                    ctypes.c_int, _P]),
    "ra_bpt_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(BptParams)]),
    "ra_bpt_fwd": (ctypes.c_int, [ctypes.POINTER(BptParams), _P, ctypes.POINTER(BptWeights), _P,
                                  ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "ra_bpt_train_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(BptParams)]),
    "ra_bpt_bwd": (ctypes.c_int, [ctypes.POINTER(BptParams), _P, ctypes.POINTER(BptWeights), _P,
                                  ctypes.POINTER(BptGrads), _P, ctypes.c_size_t, _P]),
    "ra_last_error_message": (ctypes.c_char_p, []),
    "ra_selftest_exp2": (ctypes.c_int, [_P, _P, _P, ctypes.c_longlong, _P]),
    "ra_checks_enabled": (ctypes.c_int, []),
}


def lib():
    """Load libra.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libra.so is not built: run exact_blockwise_ring_gb300.build."
                                   "build() (needs nvcc for sm_103a)")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
    return _lib


def header_symbols():
    """Names of the functions declared in include/ra.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"\b(ra_[a-z_]+)\s*\(", text)))


def _check(status):
    if status != 0:
        msg = lib().ra_last_error_message().decode(errors="replace")
        raise RaError(status, msg)


def make_params(batch, seq_len, heads, head_dim, P, block, layout="contiguous", causal=True,
                softmax_scale=0.0, n_split=0, kv_heads=0):
    if isinstance(layout, str):
        layout = LAYOUTS[layout]
    return Params(int(batch), int(seq_len), int(heads), int(head_dim), int(block), int(P),
                  int(layout), int(bool(causal)) if isinstance(causal, bool) else int(causal),
                  float(softmax_scale), int(n_split), int(kv_heads))


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_qkv(q, k, v, dout=None):
    """q (and dout) [B, L, H, D]; k, v [B, L, H_kv, D] with H_kv dividing H.  Returns
    (B, L, H, D, H_kv)."""
    ts = (q, k, v) if dout is None else (q, k, v, dout)
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v (and dout) must be contiguous 4-D CUDA bf16 tensors")
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    if (dout is not None and dout.shape != q.shape) or k.shape != v.shape or \
            k.shape[:2] != (B, L) or k.shape[3] != D or Hkv < 1 or H % Hkv:
        raise ValueError("expected q, dout [B, L, H, D] and k, v [B, L, H_kv, D], H_kv | H")
    return B, L, H, D, Hkv


class Workspace:
    """A zero-initialised device buffer reused across calls (grown on demand)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = torch.zeros(256, dtype=torch.uint8, device=self.device)

    def get(self, nbytes):
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(int(nbytes), dtype=torch.uint8, device=self.device)
        return self.buf

    def check(self, stream=None):
        """Sync the stream and raise RaError if a kernel gave up a wait."""
        _check(lib().ra_check_error(_ptr(self.buf), _stream(stream)))


_default_ws = {}


def default_workspace(device):
    key = torch.device(device).index or 0
    if key not in _default_ws:
        _default_ws[key] = Workspace(torch.device("cuda", key))
    return _default_ws[key]


def fwd_workspace_bytes(params):
    return lib().ra_fwd_workspace_bytes(ctypes.byref(params))


def bwd_workspace_bytes(params):
    return lib().ra_bwd_workspace_bytes(ctypes.byref(params))


def ra_fwd(q, k, v, P, block, layout="contiguous", causal=True, softmax_scale=0.0,
           out_dtype=torch.bfloat16, n_split=0, shard_work=False, workspace=None, stream=None,
           out=None, lse=None):
    """Forward pass through ra_fwd.  Returns (out, lse) or (out, lse, shard_work[3, P]).
    k and v may have fewer heads than q (grouped-query attention)."""
    B, L, H, D, Hkv = _check_qkv(q, k, v)
    prm = make_params(B, L, H, D, P, block, layout, causal, softmax_scale, n_split, Hkv)
    if out is None:
        out = torch.empty((B, L, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    odt = RA_FP32 if out.dtype == torch.float32 else RA_BF16
    sw = torch.empty(3 * P, dtype=torch.int64, device=q.device) if shard_work else None
    ws = workspace or default_workspace(q.device)
    need = fwd_workspace_bytes(prm)
    buf = ws.get(max(need, 256))
    _check(lib().ra_fwd(ctypes.byref(prm), _ptr(q), _ptr(k), _ptr(v), _ptr(out), odt, _ptr(lse),
                        _ptr(sw), _ptr(buf), buf.numel(), _stream(stream)))
    if shard_work:
        return out, lse, sw.view(3, P)
    return out, lse


def ra_bwd(q, k, v, out, lse, dout, P, block, layout="contiguous", causal=True,
           softmax_scale=0.0, workspace=None, stream=None, dq=None, dk=None, dv=None):
    """Backward pass through ra_bwd.  Returns (dq, dk, dv) bf16, dk and dv shaped like k."""
    B, L, H, D, Hkv = _check_qkv(q, k, v, dout)
    prm = make_params(B, L, H, D, P, block, layout, causal, softmax_scale, 0, Hkv)
    odt = RA_FP32 if out.dtype == torch.float32 else RA_BF16
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = workspace or default_workspace(q.device)
    need = bwd_workspace_bytes(prm)
    buf = ws.get(max(need, 256))
    _check(lib().ra_bwd(ctypes.byref(prm), _ptr(q), _ptr(k), _ptr(v), _ptr(out), odt, _ptr(lse),
                        _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(buf), buf.numel(),
                        _stream(stream)))
    return dq, dk, dv


def ra_bwd_stages(q, k, v, out, lse, dout, dq, dk, dv, P, block, layout="contiguous",
                  causal=True, softmax_scale=0.0, workspace=None, stream=None, between=None):
    """The backward as its three C-ABI stages (preprocess, main, finalize).

    ``between(i)`` (optional) is called before stage i (0, 1, 2) and after the last
    (i = 3), e.g. to record CUDA events around each stage."""
    B, L, H, D, Hkv = _check_qkv(q, k, v, dout)
    prm = make_params(B, L, H, D, P, block, layout, causal, softmax_scale, 0, Hkv)
    odt = RA_FP32 if out.dtype == torch.float32 else RA_BF16
    ws = workspace or default_workspace(q.device)
    buf = ws.get(max(bwd_workspace_bytes(prm), 256))
    st = _stream(stream)
    h = lib()
    if between:
        between(0)
    _check(h.ra_bwd_preprocess(ctypes.byref(prm), _ptr(out), odt, _ptr(lse), _ptr(dout),
                               _ptr(buf), buf.numel(), st))
    if between:
        between(1)
    _check(h.ra_bwd_main(ctypes.byref(prm), _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dk),
                         _ptr(dv), _ptr(buf), buf.numel(), st))
    if between:
        between(2)
    _check(h.ra_bwd_finalize(ctypes.byref(prm), _ptr(dq), _ptr(buf), buf.numel(), st))
    if between:
        between(3)
    return dq, dk, dv


def ra_merge(o_parts, lse_parts, out_dtype=torch.bfloat16, stream=None):
    """Merge partials o_parts [n, B, L, H, D] fp32 and lse_parts [n, B, H, L]."""
    n, B, L, H, D = o_parts.shape
    out = torch.empty((B, L, H, D), dtype=out_dtype, device=o_parts.device)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=o_parts.device)
    odt = RA_FP32 if out_dtype == torch.float32 else RA_BF16
    _check(lib().ra_merge(n, _ptr(o_parts.contiguous()), _ptr(lse_parts.contiguous()), B, L, H, D,
                          _ptr(out), odt, _ptr(lse), _stream(stream)))
    return out, lse


def ra_shard_work_model(seq_len, P, block, layout, causal):
    """Host closed-form work model: dict of lists (tiles, pairs, visits) per shard."""
    prm = make_params(1, seq_len, 1, 128, P, block, layout, causal)
    arr = (ctypes.c_ulonglong * (3 * P))()
    _check(lib().ra_shard_work_model(ctypes.byref(prm), arr))
    vals = list(arr)
    return {"tiles": vals[:P], "pairs": vals[P:2 * P], "visits": vals[2 * P:]}


def ra_selftest_exp2(x, stream=None):
    """Both 2^x forms of the softmax kernels on a CUDA fp32 tensor: (software, hardware)."""
    _want(x, torch.float32, "x")
    y_soft, y_hw = torch.empty_like(x), torch.empty_like(x)
    _check(lib().ra_selftest_exp2(_ptr(x), _ptr(y_soft), _ptr(y_hw), x.numel(), _stream(stream)))
    return y_soft, y_hw


def ra_selftest_timeout(workspace, timeout_us, stream=None):
    buf = workspace.get(256)
    _check(lib().ra_selftest_timeout(_ptr(buf), buf.numel(), int(timeout_us), _stream(stream)))


def _want(t, dtype, name, shape=None, device=None):
    """Raise unless t is a contiguous CUDA tensor of dtype (and shape / device)."""
    if t is None or not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if device is not None and t.device != device:
        raise ValueError("%s must be on %s" % (name, device))


def ra_linear(x, weight, bias, epilogue="bias", residual=None, workspace=None, stream=None,
              out=None):
    """out = epilogue(x weight^T + bias) through ra_linear.  x [..., in] bf16, weight
    [out, in] bf16, bias [out] fp32; "bias" / "bias_gelu" give bf16, "bias_residual" adds
    residual [..., out] bf16 and gives fp32."""
    epi = EPILOGUES[epilogue]
    n_out, n_in = weight.shape
    _want(x, torch.bfloat16, "x")
    _want(weight, torch.bfloat16, "weight")
    _want(bias, torch.float32, "bias", (n_out,))
    if x.shape[-1] != n_in:
        raise ValueError("x has %d features, weight expects %d" % (x.shape[-1], n_in))
    if epi == 2:
        _want(residual, torch.bfloat16, "residual", tuple(x.shape[:-1]) + (n_out,))
    rows = x.numel() // x.shape[-1]
    shape = tuple(x.shape[:-1]) + (n_out,)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32 if epi == 2 else torch.bfloat16,
                          device=x.device)
    ws = workspace or default_workspace(x.device)
    buf = ws.get(256)
    _check(lib().ra_linear(rows, n_in, n_out, _ptr(x), _ptr(weight), _ptr(bias), _ptr(residual),
                           epi, _ptr(out), _ptr(buf), buf.numel(), _stream(stream)))
    return out


def ra_layernorm(x, gamma, beta, eps=1e-5, out_dtype=torch.bfloat16, stream=None):
    """LayerNorm over the last dimension of fp32 x through ra_layernorm."""
    d = x.shape[-1]
    _want(x, torch.float32, "x")
    _want(gamma, torch.float32, "gamma", (d,))
    _want(beta, torch.float32, "beta", (d,))
    out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    odt = RA_FP32 if out_dtype == torch.float32 else RA_BF16
    _check(lib().ra_layernorm(x.numel() // d, d, _ptr(x), _ptr(gamma), _ptr(beta), float(eps),
                              _ptr(out), odt, _stream(stream)))
    return out


def make_bpt_params(batch, seq_len, heads, head_dim, d_ff, P, block, layout="contiguous",
                    causal=True, block_rows=0, ln_eps=0.0, n_split=0, kv_heads=0):
    return BptParams(make_params(batch, seq_len, heads, head_dim, P, block, layout, causal, 0.0,
                                 n_split, kv_heads), int(d_ff), int(block_rows), float(ln_eps))


def bpt_workspace_bytes(params):
    return lib().ra_bpt_workspace_bytes(ctypes.byref(params))


def _bpt_params_of(x, weights, heads, P, block, layout, causal, block_rows):
    """Check the layer's parameter tensors and build its ra_bpt_params_t; the number of
    key/value heads follows from wk's shape [H_kv * head_dim, d]."""
    B, L, d = x.shape
    hd = d // heads
    for n in BPT_WEIGHTS:
        if n not in weights:
            raise ValueError("missing layer parameter %r" % n)
    d_ff = weights["w1"].shape[0]
    d_kv = weights["wk"].shape[0]
    shapes = {"wq": (d, d), "wk": (d_kv, d), "wv": (d_kv, d), "wo": (d, d), "w1": (d_ff, d),
              "w2": (d, d_ff), "bq": (d,), "bk": (d_kv,), "bv": (d_kv,), "bo": (d,),
              "b1": (d_ff,), "b2": (d,), "ln1_g": (d,), "ln1_b": (d,), "ln2_g": (d,),
              "ln2_b": (d,)}
    for n in BPT_WEIGHTS:
        _want(weights[n], torch.bfloat16 if n[0] == "w" else torch.float32, n, shapes[n],
              x.device)
    if d_kv % hd or heads % (d_kv // hd):
        raise ValueError("wk has %d rows: not a divisor of the heads times head_dim %d" % (d_kv, hd))
    return make_bpt_params(B, L, heads, hd, d_ff, P, block, layout, causal, block_rows,
                           kv_heads=d_kv // hd)


def bpt_train_workspace_bytes(params):
    return lib().ra_bpt_train_workspace_bytes(ctypes.byref(params))


def ra_bpt_fwd(x, weights, heads, P, block, layout="contiguous", causal=True, block_rows=0,
               out_dtype=torch.bfloat16, workspace=None, stream=None, out=None, train=False):
    """One blockwise transformer layer forward through ra_bpt_fwd.  x [B, L, d] bf16;
    weights: dict with the names of BPT_WEIGHTS (weights bf16 [out, in], the rest fp32).
    train=True sizes the workspace for a following ra_bpt_bwd, which reuses it."""
    B, L, d = x.shape
    _want(x, torch.bfloat16, "x")
    prm = _bpt_params_of(x, weights, heads, P, block, layout, causal, block_rows)
    w = BptWeights(*[weights[n].data_ptr() for n in BPT_WEIGHTS])
    if out is None:
        out = torch.empty((B, L, d), dtype=out_dtype, device=x.device)
    odt = RA_FP32 if out.dtype == torch.float32 else RA_BF16
    ws = workspace or default_workspace(x.device)
    need = bpt_train_workspace_bytes(prm) if train else bpt_workspace_bytes(prm)
    buf = ws.get(max(need, 256))
    _check(lib().ra_bpt_fwd(ctypes.byref(prm), _ptr(x), ctypes.byref(w), _ptr(out), odt,
                            _ptr(buf), buf.numel(), _stream(stream)))
    return out


def ra_bpt_bwd(x, weights, dout, heads, P, block, layout="contiguous", causal=True,
               block_rows=0, workspace=None, stream=None):
    """Gradients of the layer through ra_bpt_bwd, after ra_bpt_fwd(..., train=True) with the
    same workspace.  Returns a dict: "x" (bf16, like x) and every name of BPT_WEIGHTS
    (fp32, shaped like the parameter)."""
    _want(x, torch.bfloat16, "x")
    _want(dout, torch.bfloat16, "dout", tuple(x.shape), x.device)
    prm = _bpt_params_of(x, weights, heads, P, block, layout, causal, block_rows)
    w = BptWeights(*[weights[n].data_ptr() for n in BPT_WEIGHTS])
    grads = {"x": torch.empty_like(x)}
    for n in BPT_WEIGHTS:
        grads[n] = torch.empty(weights[n].shape, dtype=torch.float32, device=x.device)
    g = BptGrads(grads["x"].data_ptr(), *[grads[n].data_ptr() for n in BPT_WEIGHTS])
    ws = workspace or default_workspace(x.device)
    need = bpt_train_workspace_bytes(prm)
    if ws.buf.numel() < need:
        raise ValueError("the workspace does not hold the forward's state: run ra_bpt_fwd "
                         "with train=True and the same workspace first")
    _check(lib().ra_bpt_bwd(ctypes.byref(prm), _ptr(x), ctypes.byref(w), _ptr(dout),
                            ctypes.byref(g), _ptr(ws.buf), ws.buf.numel(), _stream(stream)))
    return grads


class BptLayer(torch.autograd.Function):
    """autograd wrapper of one blockwise transformer layer: forward = ra_bpt_fwd (train
    mode, its own workspace kept for the backward), backward = ra_bpt_bwd.  Call as
    BptLayer.apply(x, (heads, P, block, layout, causal, block_rows), *weights in the order
    of BPT_WEIGHTS); weight gradients come back in fp32 and are cast to the weights'
    dtypes."""

    @staticmethod
    def forward(ctx, x, cfg, *params):
        heads, P, block, layout, causal, block_rows = cfg
        weights = dict(zip(BPT_WEIGHTS, params))
        ws = Workspace(x.device)
        out = ra_bpt_fwd(x, weights, heads, P, block, layout, causal, block_rows, workspace=ws,
                         train=True)
        ctx.save_for_backward(x, *params)
        ctx.cfg, ctx.ws = cfg, ws
        return out

    @staticmethod
    def backward(ctx, dout):
        x, *params = ctx.saved_tensors
        heads, P, block, layout, causal, block_rows = ctx.cfg
        weights = dict(zip(BPT_WEIGHTS, params))
        g = ra_bpt_bwd(x, weights, dout.contiguous(), heads, P, block, layout, causal,
                       block_rows, workspace=ctx.ws)
        return (g["x"], None) + tuple(g[n].to(weights[n].dtype) for n in BPT_WEIGHTS)


class RingAttention(torch.autograd.Function):
    """autograd wrapper: forward = ra_fwd, backward = ra_bwd (lse saved, scores
    recomputed)."""

    @staticmethod
    def forward(ctx, q, k, v, P, block, layout, causal, softmax_scale):
        out, lse = ra_fwd(q, k, v, P, block, layout, causal, softmax_scale)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.cfg = (P, block, layout, causal, softmax_scale)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        P, block, layout, causal, scale = ctx.cfg
        dq, dk, dv = ra_bwd(q, k, v, out, lse, dout.contiguous(), P, block, layout, causal, scale)
        return dq, dk, dv, None, None, None, None, None


def ring_attention(q, k, v, P, block, layout="contiguous", causal=True, softmax_scale=0.0):
    return RingAttention.apply(q, k, v, P, block, layout, causal, softmax_scale)
