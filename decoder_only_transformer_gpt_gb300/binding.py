"""Thin ctypes binding of the C ABI (include/gpt.h, include/gpt_kernels.h).

Argument marshalling only: every step of the forward pass runs in the CUDA
library. PyTorch supplies device memory and streams. If the library has not
been built, or a call fails, this module raises; there is no fallback.
"""
import ctypes
import os
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpt_gb300.so")

GPT_OK, GPT_EINVAL, GPT_ECONFIG, GPT_ESEQ, GPT_ETOKEN, GPT_ECUDA, GPT_ENOMEM, GPT_EDEVICE, GPT_EUNSUPPORTED = range(9)
# parameters of gpt_grad, in the library's order; the per-block ones take a layer index
GRAD_PARAMS = ("wte", "wpe", "lnf_g", "lnf_b", "ln1_g", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
               "ln2_g", "ln2_b", "fc_w", "fc_b", "mp_w", "mp_b", "head")
EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESID, EPI_F32 = range(4)

_fp = ctypes.POINTER(ctypes.c_float)


class GptConfig(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int32), ("C", ctypes.c_int32), ("H", ctypes.c_int32), ("L", ctypes.c_int32),
                ("ctx", ctypes.c_int32), ("ffn", ctypes.c_int32), ("norm_mode", ctypes.c_int32),
                ("final_ln", ctypes.c_int32), ("gelu", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("ln_eps", ctypes.c_float), ("max_tokens", ctypes.c_int64), ("untied_head", ctypes.c_int32)]


class GptLayerWeights(ctypes.Structure):
    _fields_ = [(n, _fp) for n in ("ln1_g", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
                                   "ln2_g", "ln2_b", "fc_w", "fc_b", "mp_w", "mp_b")]


class GptWeights(ctypes.Structure):
    _fields_ = [("wte", _fp), ("wpe", _fp), ("layers", ctypes.POINTER(GptLayerWeights)),
                ("lnf_g", _fp), ("lnf_b", _fp), ("head", _fp)]


class GptError(RuntimeError):
    def __init__(self, code: int, where: str, lib=None):
        msg = f"{where}: status {code}"
        if lib is not None:
            msg += f" ({lib.gpt_strerror(code).decode()})"
            detail = lib.gpt_last_error_detail().decode()
            if detail:
                msg += f" [{detail}]"
        super().__init__(msg)
        self.code = code


_LIB = None


def load(path: str = LIB_PATH):
    """Load the built library; raise if it is missing (no fallback path exists)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sigs = {
        "gpt_create": (ctypes.c_int, [ctypes.POINTER(GptConfig), ctypes.POINTER(GptWeights), ctypes.POINTER(vp)]),
        "gpt_forward": (ctypes.c_int, [vp, vp, vp, i32, i32, vp, vp, vp]),
        "gpt_forward_host": (ctypes.c_int, [vp, vp, vp, i32, i32, vp, vp, vp]),
        "gpt_status": (ctypes.c_int, [vp, vp]),
        "gpt_destroy": (None, [vp]),
        "gpt_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "gpt_last_error_detail": (ctypes.c_char_p, []),
        "gpt_param_count": (i64, [ctypes.POINTER(GptConfig)]),
        "gpt_time_step": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp]),
        "gpt_last_launch_count": (ctypes.c_int, [vp]),
        "gpt_last_probe_hits": (ctypes.c_int, [vp]),
        "gpt_debug_expire_waits": (ctypes.c_int, [vp, i64]),
        "gpt_kv_reserve": (ctypes.c_int, [vp, i32]),
        "gpt_prefill": (ctypes.c_int, [vp, vp, i32, i32, vp, vp]),
        "gpt_decode_step": (ctypes.c_int, [vp, vp, i32, i32, vp, vp]),
        "gpt_sample": (ctypes.c_int, [vp, i32, i32, ctypes.c_float, i32, ctypes.c_float, vp, vp, vp]),
        "gpt_backward": (ctypes.c_int, [vp, vp, vp, i32, i32, vp, vp]),
        "gpt_grad": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(i64)]),
        "gpt_grad_copy": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp]),
        "gpt_adamw_step": (ctypes.c_int, [vp, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_float, vp]),
        "gpt_master_copy": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp]),
        "gptk_gemm": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
        "gptk_gemm_pair": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
        "gptk_attention": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, i32, vp]),
        "gptk_attention_lse": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, vp]),
        "gptk_attention_bwd": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]),
        "gptk_layernorm": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, ctypes.c_float, i32, vp]),
        "gptk_embed": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]),
        "gptk_lmhead_ce": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]),
        "gptk_lmhead_ce_noalloc": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, i32, vp, vp]),
        "gptk_mean": (ctypes.c_int, [vp, i32, vp, vp]),
        "gptk_status": (ctypes.c_int, [vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(rc: int, where: str):
    if rc != GPT_OK:
        raise GptError(rc, where, _LIB)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_config(cfg, max_tokens: int) -> GptConfig:
    return GptConfig(V=cfg.V, C=cfg.C, H=cfg.H, L=cfg.L, ctx=cfg.ctx, ffn=cfg.ffn, norm_mode=cfg.norm_mode,
                     final_ln=cfg.final_ln, gelu=cfg.gelu, dtype=cfg.dtype, ln_eps=cfg.ln_eps,
                     max_tokens=max_tokens, untied_head=getattr(cfg, "untied_head", 0))


def param_count(cfg) -> int:
    lib = load()
    c = make_config(cfg, 1)
    return int(lib.gpt_param_count(ctypes.byref(c)))


class GPTModel:
    """A model handle: gpt_create on construction, gpt_destroy on close()."""

    def __init__(self, cfg, weights: dict, max_tokens: int):
        self.lib = load()
        self.cfg = cfg
        self.max_tokens = max_tokens
        c = make_config(cfg, max_tokens)
        keep = []

        def fp(a):
            if a is None:
                return None
            arr = np.ascontiguousarray(a, dtype=np.float32)
            keep.append(arr)
            return arr.ctypes.data_as(_fp)

        layers = (GptLayerWeights * max(1, cfg.L))()
        for i, p in enumerate(weights["layers"]):
            layers[i] = GptLayerWeights(**{name: fp(p[name]) for name, _ in GptLayerWeights._fields_})
        w = GptWeights(wte=fp(weights["wte"]), wpe=fp(weights["wpe"]), layers=layers,
                       lnf_g=fp(weights.get("lnf_g")), lnf_b=fp(weights.get("lnf_b")),
                       head=fp(weights.get("head")))
        h = ctypes.c_void_p()
        _check(self.lib.gpt_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)), "gpt_create")
        self.handle = h
        del keep

    def forward(self, ids, targets=None, loss=None, logits=None, stream=None, check: bool = True):
        """Device tensors in, device tensors out (asynchronous unless check=True)."""
        B, T = ids.shape
        _check(self.lib.gpt_forward(self.handle, _ptr(ids), _ptr(targets), B, T, _ptr(loss), _ptr(logits),
                                    _stream(stream)), "gpt_forward")
        if check:
            self.status(stream)

    def forward_host(self, ids: np.ndarray, targets: Optional[np.ndarray] = None, want_logits: bool = False,
                     stream=None):
        """Host buffers in and out; returns (loss or None, logits or None)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        B, T = ids.shape
        tg = None if targets is None else np.ascontiguousarray(targets, dtype=np.int32)
        loss = ctypes.c_float(0.0)
        logits = np.empty((B, T, self.cfg.V), np.float32) if want_logits else None
        rc = self.lib.gpt_forward_host(self.handle, ids.ctypes.data, None if tg is None else tg.ctypes.data, B, T,
                                       ctypes.addressof(loss) if tg is not None else None,
                                       None if logits is None else logits.ctypes.data, _stream(stream))
        _check(rc, "gpt_forward_host")
        return (float(loss.value) if tg is not None else None), logits

    def forward_host_ptrs(self, ids_ptr: int, tg_ptr: Optional[int], B: int, T: int, loss_ptr: int,
                          stream=None) -> None:
        """The host-buffer entry with raw (e.g. pinned) host pointers."""
        _check(self.lib.gpt_forward_host(self.handle, ids_ptr, tg_ptr, B, T, loss_ptr, None, _stream(stream)),
               "gpt_forward_host")

    def kv_reserve(self, max_batch: int) -> None:
        """Allocate the key/value cache for up to max_batch sequences of ctx tokens."""
        _check(self.lib.gpt_kv_reserve(self.handle, max_batch), "gpt_kv_reserve")

    def prefill(self, ids, logits=None, stream=None) -> None:
        """Forward over prompts ids [B, T] (device int32) that fills the cache; logits [B, V] of the last tokens."""
        B, T = ids.shape
        _check(self.lib.gpt_prefill(self.handle, _ptr(ids), B, T, _ptr(logits), _stream(stream)), "gpt_prefill")

    def decode_step(self, ids, pos: int, logits, stream=None) -> None:
        """Append ids [B] (device int32) at position pos; logits [B, V] of the next token."""
        _check(self.lib.gpt_decode_step(self.handle, _ptr(ids), ids.shape[0], pos, _ptr(logits), _stream(stream)),
               "gpt_decode_step")

    def backward(self, ids, targets, loss=None, stream=None, check: bool = True) -> None:
        """Forward, loss and the gradient of every parameter (device int32 ids / targets [B, T])."""
        B, T = ids.shape
        _check(self.lib.gpt_backward(self.handle, _ptr(ids), _ptr(targets), B, T, _ptr(loss), _stream(stream)),
               "gpt_backward")
        if check:
            self.status(stream)

    def grad(self, name: str, layer: int = -1, stream=None):
        """A copy of one parameter's gradient from the last backward, as a device fp32 tensor shaped like it."""
        import torch
        param = GRAD_PARAMS.index(name)
        ptr, n = ctypes.c_void_p(), ctypes.c_int64()
        _check(self.lib.gpt_grad(self.handle, param, layer, ctypes.byref(ptr), ctypes.byref(n)), "gpt_grad")
        c = self.cfg
        shapes = {"wte": (c.V, c.C), "head": (c.V, c.C), "wpe": (c.ctx, c.C), "attn_w": (3 * c.C, c.C), "attn_b": (3 * c.C,),
                  "proj_w": (c.C, c.C), "fc_w": (c.ffn, c.C), "fc_b": (c.ffn,), "mp_w": (c.C, c.ffn)}
        out = torch.empty(shapes.get(name, (c.C,)), dtype=torch.float32, device="cuda")
        assert out.numel() == n.value
        _check(self.lib.gpt_grad_copy(self.handle, param, layer, _ptr(out), _stream(stream)), "gpt_grad_copy")
        return out

    def adamw_step(self, lr: float, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                   weight_decay: float = 0.0, stream=None) -> None:
        """One AdamW update of the model's weights from the last backward's gradients."""
        _check(self.lib.gpt_adamw_step(self.handle, lr, beta1, beta2, eps, weight_decay, _stream(stream)),
               "gpt_adamw_step")

    def master(self, name: str, layer: int = -1, stream=None):
        """A copy of one parameter's fp32 master weight (after an AdamW step)."""
        g = self.grad(name, layer, stream)            # same shape and numel
        _check(self.lib.gpt_master_copy(self.handle, GRAD_PARAMS.index(name), layer, _ptr(g), _stream(stream)),
               "gpt_master_copy")
        return g

    def grads(self, stream=None) -> dict:
        """Every gradient, keyed like the weight dict ("layers" a list of per-block dicts)."""
        g = {k: self.grad(k, -1, stream) for k in GRAD_PARAMS[:4]}
        if getattr(self.cfg, "untied_head", 0):
            g["head"] = self.grad("head", -1, stream)
        g["layers"] = [{k: self.grad(k, l, stream) for k in GRAD_PARAMS[4:16]} for l in range(self.cfg.L)]
        return g

    def status(self, stream=None):
        _check(self.lib.gpt_status(self.handle, _stream(stream)), "gpt_status")

    def debug_expire_waits(self, limit_cycles: int) -> None:
        """Arm the failure-detection check for the next forward (see gpt_debug_expire_waits)."""
        _check(self.lib.gpt_debug_expire_waits(self.handle, limit_cycles), "gpt_debug_expire_waits")

    def close(self):
        if getattr(self, "handle", None):
            self.lib.gpt_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- per-step entries

def sample(logits, uniform, ids_out, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0, stream=None):
    """Next-token ids [B] from logits [B, V] (device tensors); uniform [B] in [0, 1) from the caller."""
    lib = load()
    B, V = logits.shape
    _check(lib.gpt_sample(_ptr(logits), B, V, temperature, top_k, top_p, _ptr(uniform), _ptr(ids_out),
                          _stream(stream)), "gpt_sample")


def gemm(A, W, bias, out, epilogue: int, stream=None):
    lib = load()
    M, K = A.shape
    N = W.shape[0]
    dtype = 1 if A.dtype.is_floating_point and A.element_size() == 2 else 0
    _check(lib.gptk_gemm(_ptr(A), _ptr(W), _ptr(bias), _ptr(out), M, N, K, epilogue, dtype, _stream(stream)),
           "gptk_gemm")


def gemm_pair(A, W, bias, out, ksplit: int = 0, epilogue: int = EPI_BIAS_RESID, stream=None):
    lib = load()
    M, K = A.shape
    N = W.shape[0]
    _check(lib.gptk_gemm_pair(_ptr(A), _ptr(W), _ptr(bias), _ptr(out), M, N, K, epilogue, ksplit, _stream(stream)),
           "gptk_gemm_pair")


def attention(qkv, y, H: int, stream=None):
    lib = load()
    B, T, C3 = qkv.shape
    D = C3 // 3 // H
    dtype = 1 if qkv.element_size() == 2 else 0
    _check(lib.gptk_attention(_ptr(qkv), _ptr(y), B, T, H, D, dtype, _stream(stream)), "gptk_attention")


def attention_lse(qkv, y, lse2, H: int, stream=None):
    """bf16 attention that also writes each query row's base-2 log-sum-exp, lse2 fp32 [B*H*T]."""
    lib = load()
    B, T, C3 = qkv.shape
    D = C3 // 3 // H
    _check(lib.gptk_attention_lse(_ptr(qkv), _ptr(y), _ptr(lse2), B, T, H, D, _stream(stream)), "gptk_attention_lse")


def attention_bwd(qkv, y, dy, lse2, dqkv, H: int, stream=None):
    """dqkv [B, T, 3C] bf16 from qkv, the attention output y, its gradient dy and lse2 of attention_lse."""
    lib = load()
    B, T, C3 = qkv.shape
    D = C3 // 3 // H
    _check(lib.gptk_attention_bwd(_ptr(qkv), _ptr(y), _ptr(dy), _ptr(lse2), _ptr(dqkv), B, T, H, D,
                                  _stream(stream)), "gptk_attention_bwd")


def layernorm(x, g, b, out, out_f32=None, eps: float = 1e-5, stream=None):
    lib = load()
    M, C = x.shape
    dtype = 1 if out.element_size() == 2 else 0
    _check(lib.gptk_layernorm(_ptr(x), _ptr(g), _ptr(b), _ptr(out), _ptr(out_f32), M, C, eps, dtype,
                              _stream(stream)), "gptk_layernorm")


def embed(ids, wte, wpe, x, stream=None):
    lib = load()
    B, T = ids.shape
    V, C = wte.shape
    dtype = 1 if wte.element_size() == 2 else 0
    _check(lib.gptk_embed(_ptr(ids), _ptr(wte), _ptr(wpe), _ptr(x), B, T, C, V, dtype, _stream(stream)),
           "gptk_embed")


def lmhead_ce(h, wte, targets, nll, logits=None, stream=None):
    lib = load()
    M, C = h.shape
    V = wte.shape[0]
    dtype = 1 if h.element_size() == 2 else 0
    _check(lib.gptk_lmhead_ce(_ptr(h), _ptr(wte), _ptr(targets), _ptr(nll), _ptr(logits), M, V, C, dtype,
                              _stream(stream)), "gptk_lmhead_ce")


def lmhead_ce_noalloc(h, wte, targets, nll, err=None, stream=None):
    """Head + cross-entropy with no device allocation: for callers that cannot
    allocate while they run (a fixed start-up memory budget, a caching allocator
    that owns the free memory, or a loop that must not synchronise). Uses the
    library's fixed 8 MiB scratch array; `err` is an optional device int32."""
    lib = load()
    M, C = h.shape
    V = wte.shape[0]
    _check(lib.gptk_lmhead_ce_noalloc(_ptr(h), _ptr(wte), _ptr(targets), _ptr(nll), M, V, C, _ptr(err),
                                      _stream(stream)), "gptk_lmhead_ce_noalloc")


def mean(nll, loss, stream=None):
    lib = load()
    _check(lib.gptk_mean(_ptr(nll), nll.numel(), _ptr(loss), _stream(stream)), "gptk_mean")


def status(stream=None):
    lib = load()
    _check(lib.gptk_status(_stream(stream)), "gptk_status")
