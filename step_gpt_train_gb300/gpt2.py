"""Python binding of the C ABI in include/gpt2.h and include/gpt2_ops.h.

Argument marshalling only: every step of the training step runs in the CUDA
library (libgpt2.so). PyTorch supplies device memory (one uint8 workspace
tensor) and the CUDA stream. There is no fallback: if the library is not
built, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint64, c_void_p, c_char_p

import numpy as np

from . import _build

MODE_FP32 = 0
MODE_BF16 = 1

GPT2_OK = 0
STATUS_NAMES = {
    0: "GPT2_OK", -1: "GPT2_ERR_ARG", -2: "GPT2_ERR_STATE", -3: "GPT2_ERR_TOKEN_RANGE",
    -4: "GPT2_ERR_NONFINITE", -5: "GPT2_ERR_TIMEOUT", -6: "GPT2_ERR_CUDA", -7: "GPT2_ERR_WORKSPACE",
}

TENSOR_PARAM, TENSOR_MASTER, TENSOR_GRAD, TENSOR_ADAM_M, TENSOR_ADAM_V = range(5)
FP8_E4M3, FP8_E5M2 = 0, 1  # the FP8 formats of gpt2_op_quantize_fp8 / gpt2_op_matmul_fp8

FAMILIES = ["encoder_forward", "layernorm_forward", "matmul", "attention_forward", "residual_forward",
            "gelu_forward", "classifier", "loss_mean", "layernorm_backward", "gelu_backward",
            "bias_backward", "attention_backward", "residual_backward", "encoder_backward", "adamw",
            "grad_colsum", "fp8_quant"]

# FP8 linear layers (gpt2_set_fp8)
FP8_QKV, FP8_MLP, FP8_HEAD = 1, 2, 4
FP8_ALL = FP8_QKV | FP8_MLP | FP8_HEAD

WORKSPACE_ALIGN = 1024


class GPT2Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({_strerror(status)})")


class gpt2_config(ctypes.Structure):
    _fields_ = [("n_layer", c_int32), ("n_embd", c_int32), ("n_head", c_int32), ("vocab", c_int32),
                ("vocab_padded", c_int32), ("max_T", c_int32), ("max_B", c_int32), ("mode", c_int32)]


class gpt2_adamw_config(ctypes.Structure):
    _fields_ = [("lr", c_float), ("beta1", c_float), ("beta2", c_float), ("eps", c_float),
                ("weight_decay", c_float), ("t", c_int32), ("grad_scale", c_float), ("max_grad_norm", c_float),
                ("decay_mask", c_int32)]


_lib = None

# name -> (restype, argtypes)
_SIGNATURES = {
    "gpt2_workspace_bytes": (c_int, [POINTER(gpt2_config), POINTER(c_size_t)]),
    "gpt2_init": (c_int, [POINTER(c_void_p), POINTER(gpt2_config), c_uint64, c_void_p, c_size_t, c_void_p]),
    "gpt2_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, POINTER(c_float)]),
    "gpt2_backward": (c_int, [c_void_p]),
    "gpt2_adamw_step": (c_int, [c_void_p, c_float, c_float, c_float, c_float, c_float, c_int]),
    "gpt2_destroy": (c_int, [c_void_p]),
    "gpt2_set_grad_accumulation": (c_int, [c_void_p, c_int]),
    "gpt2_fp8_workspace_bytes": (c_int, [POINTER(gpt2_config), c_int, POINTER(c_size_t)]),
    "gpt2_set_fp8": (c_int, [c_void_p, c_int, c_void_p, c_size_t]),
    "gpt2_zero_grad": (c_int, [c_void_p]),
    "gpt2_grad_norm": (c_int, [c_void_p, POINTER(c_float)]),
    "gpt2_adamw_step_ex": (c_int, [c_void_p, POINTER(gpt2_adamw_config)]),
    "gpt2_adamw_step_shard": (c_int, [c_void_p, POINTER(gpt2_adamw_config), ctypes.c_int64, ctypes.c_int64]),
    "gpt2_grad_sumsq_range": (c_int, [c_void_p, ctypes.c_int64, ctypes.c_int64, POINTER(ctypes.c_float)]),
    "gpt2_flat_params": (c_int64, [c_void_p]),
    "gpt2_step": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, POINTER(gpt2_adamw_config), POINTER(c_float)]),
    "gpt2_step_host": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, POINTER(gpt2_adamw_config),
                               POINTER(c_float)]),
    "gpt2_lr_cosine": (c_float, [c_int, c_int, c_int, c_float, c_float]),
    "gpt2_strerror": (c_char_p, [c_int]),
    "gpt2_num_tensors": (c_int, [c_void_p]),
    "gpt2_tensor_info": (c_int, [c_void_p, c_int, POINTER(c_char_p), POINTER(c_int64)]),
    "gpt2_copy_tensor": (c_int, [c_void_p, c_int, c_int, c_void_p]),
    "gpt2_load_tensor": (c_int, [c_void_p, c_int, c_void_p]),
    "gpt2_copy_losses": (c_int, [c_void_p, c_void_p]),
    "gpt2_num_params": (c_int64, [c_void_p]),
    "gpt2_launch_count": (c_int64, [c_void_p]),
    "gpt2_family_stats": (c_int, [c_void_p, c_int, POINTER(c_int64), POINTER(c_int64), POINTER(c_double)]),
    "gpt2_set_timing": (c_int, [c_void_p, c_int]),
    "gpt2_family_time": (c_int, [c_void_p, c_int, POINTER(c_double)]),
    "gpt2_reset_stats": (c_int, [c_void_p]),
    # gpt2_ops.h
    "gpt2_debug_set_wait_limit": (c_int, [c_int64]),
    "gpt2_debug_stall_matmul": (c_int, [c_int]),
    "gpt2_debug_matmul_pair": (c_int, [c_int]),
    "gpt2_op_encoder_forward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                        c_void_p, c_void_p]),
    "gpt2_op_encoder_backward_scratch": (c_size_t, [c_int, c_int, c_int]),
    "gpt2_op_encoder_backward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                         c_void_p, c_size_t, c_void_p]),
    "gpt2_op_layernorm_forward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                          c_int, c_void_p]),
    "gpt2_op_layernorm_backward_scratch": (c_size_t, [c_int, c_int]),
    "gpt2_op_layernorm_backward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "gpt2_op_residual_layernorm_forward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                   c_void_p, c_void_p, c_int, c_int, c_void_p]),
    "gpt2_op_layernorm_backward_residual": (c_int, [c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                                    c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p,
                                                    c_size_t, c_void_p]),
    "gpt2_op_matmul_scratch": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "gpt2_op_matmul": (c_int, [c_int, c_void_p, c_int, c_void_p, c_int, c_void_p, c_int, c_void_p, c_int, c_int,
                               c_int, c_void_p, c_size_t, c_void_p, c_void_p]),
    "gpt2_op_matmul_gelu": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                    c_void_p, c_void_p]),
    "gpt2_op_quantize_fp8_scratch": (c_size_t, []),
    "gpt2_op_quantize_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int, c_void_p, c_size_t, c_void_p]),
    "gpt2_op_quantize_fp8_transpose": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                               c_void_p]),
    "gpt2_op_matmul_fp8_scratch": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "gpt2_op_matmul_fp8_ex": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p, c_int, c_void_p,
                                      c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_size_t,
                                      c_void_p, c_void_p]),
    "gpt2_op_matmul_fp8": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                   c_int, c_int, c_void_p, c_void_p]),
    "gpt2_op_matmul_gelu_backward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                             c_void_p, c_void_p]),
    "gpt2_op_matmul_gelu_backward_bias_scratch": (c_size_t, [c_int, c_int]),
    "gpt2_op_matmul_gelu_backward_bias": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                                  c_int, c_int, c_void_p, c_size_t, c_void_p, c_void_p]),
    "gpt2_op_attention_forward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                          c_void_p]),
    "gpt2_op_attention_backward_scratch": (c_size_t, [c_int, c_int, c_int]),
    "gpt2_op_attention_backward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                           c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "gpt2_op_gelu_forward": (c_int, [c_int, c_void_p, c_void_p, c_int64, c_void_p]),
    "gpt2_op_gelu_backward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_int64, c_void_p]),
    "gpt2_op_residual_forward": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_int64, c_void_p]),
    "gpt2_op_residual_backward": (c_int, [c_int, c_void_p, c_void_p, c_int64, c_void_p]),
    "gpt2_op_bias_backward_scratch": (c_size_t, [c_int, c_int]),
    "gpt2_op_bias_backward": (c_int, [c_int, c_void_p, c_void_p, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "gpt2_op_bias_backward_noalloc": (c_int, [c_int, c_void_p, c_void_p, c_int, c_int, c_void_p]),
    "gpt2_op_classifier": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_float, c_void_p,
                                   c_void_p]),
    "gpt2_op_mean_loss": (c_int, [c_void_p, c_void_p, c_int, c_void_p]),
    "gpt2_op_adamw": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_float, c_float, c_float,
                              c_float, c_float, c_int, c_void_p]),
}


def library_path() -> str:
    return _build.LIB


def load_library(build: bool = False) -> ctypes.CDLL:
    """Load libgpt2.so (building it first if `build`). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if build:
        _build.build()
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"the CUDA library {path} is not built; run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _strerror(status: int) -> str:
    try:
        return load_library().gpt2_strerror(status).decode()
    except Exception:
        return "?"


def check(status: int, what: str = "gpt2") -> None:
    if status != GPT2_OK:
        raise GPT2Error(status, what)


def make_config(n_layer, n_embd, n_head, vocab, vocab_padded, max_T, max_B, mode) -> gpt2_config:
    return gpt2_config(n_layer, n_embd, n_head, vocab, vocab_padded, max_T, max_B, mode)


# ---------------------------------------------------------------- C-ABI functions, same names

def gpt2_workspace_bytes(cfg: gpt2_config) -> int:
    out = c_size_t(0)
    check(load_library().gpt2_workspace_bytes(ctypes.byref(cfg), ctypes.byref(out)), "gpt2_workspace_bytes")
    return out.value


def gpt2_init(cfg: gpt2_config, seed: int, workspace_ptr: int, workspace_bytes: int, stream_ptr: int) -> c_void_p:
    h = c_void_p()
    check(load_library().gpt2_init(ctypes.byref(h), ctypes.byref(cfg), seed, workspace_ptr, workspace_bytes,
                                   stream_ptr), "gpt2_init")
    return h


def gpt2_forward(h, tokens_ptr: int, targets_ptr: int | None, B: int, T: int) -> float | None:
    loss = c_float(0.0)
    check(load_library().gpt2_forward(h, tokens_ptr, targets_ptr, B, T,
                                      ctypes.byref(loss) if targets_ptr else None), "gpt2_forward")
    return float(loss.value) if targets_ptr else None


def gpt2_backward(h) -> None:
    check(load_library().gpt2_backward(h), "gpt2_backward")


def gpt2_adamw_step(h, lr, beta1, beta2, eps, weight_decay, t) -> None:
    check(load_library().gpt2_adamw_step(h, lr, beta1, beta2, eps, weight_decay, t), "gpt2_adamw_step")


def gpt2_destroy(h) -> None:
    check(load_library().gpt2_destroy(h), "gpt2_destroy")


# ---------------------------------------------------------------- convenience wrapper

class GPT2:
    """One model in a torch-allocated workspace on the current CUDA device.

    cfg: dict with n_layer, n_embd, n_head, vocab, vocab_padded, max_T, max_B, mode.
    """

    def __init__(self, cfg: dict, seed: int, stream=None):
        import torch
        self.lib = load_library()
        self.cfg = make_config(*(int(cfg[k]) for k in ("n_layer", "n_embd", "n_head", "vocab", "vocab_padded",
                                                       "max_T", "max_B", "mode")))
        self.bytes = gpt2_workspace_bytes(self.cfg)
        self._ws = torch.empty(self.bytes + WORKSPACE_ALIGN, dtype=torch.uint8, device="cuda")
        base = self._ws.data_ptr()
        self.ws_ptr = (base + WORKSPACE_ALIGN - 1) // WORKSPACE_ALIGN * WORKSPACE_ALIGN
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.h = gpt2_init(self.cfg, seed, self.ws_ptr, self.bytes, self.stream.cuda_stream)
        self.names, self.shapes = [], []
        for i in range(self.lib.gpt2_num_tensors(self.h)):
            name = c_char_p()
            shape = (c_int64 * 2)()
            check(self.lib.gpt2_tensor_info(self.h, i, ctypes.byref(name), shape), "gpt2_tensor_info")
            self.names.append(name.value.decode())
            self.shapes.append((shape[0],) if shape[1] == 1 else (shape[0], shape[1]))

    def close(self):
        if getattr(self, "h", None):
            gpt2_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, tokens, targets=None):
        """tokens/targets: int32 CUDA tensors [B, T] (contiguous)."""
        B, T = tokens.shape
        return gpt2_forward(self.h, tokens.data_ptr(), targets.data_ptr() if targets is not None else None, B, T)

    def backward(self):
        gpt2_backward(self.h)

    def adamw_step(self, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, t=1, grad_scale=None,
                   max_grad_norm=None, decay_mask=None):
        """gpt2_adamw_step, or gpt2_adamw_step_ex when any of grad_scale,
        max_grad_norm or decay_mask is given."""
        if grad_scale is None and max_grad_norm is None and decay_mask is None:
            gpt2_adamw_step(self.h, lr, beta1, beta2, eps, weight_decay, t)
            return
        c = gpt2_adamw_config(lr, beta1, beta2, eps, weight_decay, t, 1.0 if grad_scale is None else grad_scale,
                              0.0 if max_grad_norm is None else max_grad_norm, int(bool(decay_mask)))
        check(self.lib.gpt2_adamw_step_ex(self.h, ctypes.byref(c)), "gpt2_adamw_step_ex")

    def step(self, tokens, targets, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, t=1, grad_scale=1.0,
             max_grad_norm=0.0, decay_mask=False) -> float:
        """gpt2_step: forward, backward and AdamW as one captured CUDA graph; returns the mean loss.
        tokens/targets: int32 CUDA tensors [B, T] (contiguous)."""
        B, T = tokens.shape
        c = gpt2_adamw_config(lr, beta1, beta2, eps, weight_decay, t, grad_scale, max_grad_norm,
                              int(bool(decay_mask)))
        loss = c_float(0.0)
        check(self.lib.gpt2_step(self.h, tokens.data_ptr(), targets.data_ptr(), B, T, ctypes.byref(c),
                                 ctypes.byref(loss)), "gpt2_step")
        return loss.value

    def step_host(self, tokens, targets, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, t=1,
                  grad_scale=1.0, max_grad_norm=0.0, decay_mask=False) -> float:
        """gpt2_step_host: gpt2_step with the batch in host memory, copied to the device
        by the library. tokens/targets: int32 CPU tensors [B, T] (contiguous; pinned
        for asynchronous copies)."""
        B, T = tokens.shape
        c = gpt2_adamw_config(lr, beta1, beta2, eps, weight_decay, t, grad_scale, max_grad_norm,
                              int(bool(decay_mask)))
        loss = c_float(0.0)
        check(self.lib.gpt2_step_host(self.h, tokens.data_ptr(), targets.data_ptr(), B, T, ctypes.byref(c),
                                      ctypes.byref(loss)), "gpt2_step_host")
        return loss.value

    def adamw_step_shard(self, begin, count, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, t=1,
                         grad_scale=1.0, decay_mask=False):
        """gpt2_adamw_step_shard: AdamW on the flat parameter elements [begin, begin + count)."""
        c = gpt2_adamw_config(lr, beta1, beta2, eps, weight_decay, t, grad_scale, 0.0, int(bool(decay_mask)))
        check(self.lib.gpt2_adamw_step_shard(self.h, ctypes.byref(c), int(begin), int(count)), "gpt2_adamw_step_shard")

    def grad_sumsq_range(self, begin, count) -> float:
        """gpt2_grad_sumsq_range: sum of squares of the gradient elements [begin, begin + count)."""
        out = ctypes.c_float(0.0)
        check(self.lib.gpt2_grad_sumsq_range(self.h, int(begin), int(count), ctypes.byref(out)),
              "gpt2_grad_sumsq_range")
        return out.value

    def set_fp8(self, mask: int) -> None:
        """Run the linears in mask (FP8_QKV | FP8_MLP | FP8_HEAD) with FP8
        operands; 0 returns every matmul to bf16. Allocates the codes'
        workspace (torch, on this device) and keeps it with the model."""
        import torch
        n = ctypes.c_size_t(0)
        check(self.lib.gpt2_fp8_workspace_bytes(ctypes.byref(self.cfg), int(mask), ctypes.byref(n)),
              "gpt2_fp8_workspace_bytes")
        if mask:
            self._ws8 = torch.empty(n.value + WORKSPACE_ALIGN, dtype=torch.uint8, device="cuda")
            ptr = (self._ws8.data_ptr() + WORKSPACE_ALIGN - 1) // WORKSPACE_ALIGN * WORKSPACE_ALIGN
        else:
            ptr = None
        check(self.lib.gpt2_set_fp8(self.h, int(mask), ptr, n.value), "gpt2_set_fp8")
        if not mask:
            self._ws8 = None
        self.fp8_bytes = n.value

    def set_grad_accumulation(self, on: bool) -> None:
        check(self.lib.gpt2_set_grad_accumulation(self.h, int(bool(on))), "gpt2_set_grad_accumulation")

    def zero_grad(self) -> None:
        check(self.lib.gpt2_zero_grad(self.h), "gpt2_zero_grad")

    def grad_norm(self) -> float:
        v = c_float()
        check(self.lib.gpt2_grad_norm(self.h, ctypes.byref(v)), "gpt2_grad_norm")
        return v.value

    def tensor(self, i: int, kind: int = TENSOR_MASTER) -> np.ndarray:
        out = np.empty(self.shapes[i], dtype=np.float32)
        check(self.lib.gpt2_copy_tensor(self.h, i, kind, out.ctypes.data), "gpt2_copy_tensor")
        return out

    def tensors(self, kind: int = TENSOR_MASTER) -> dict:
        return {n: self.tensor(i, kind) for i, n in enumerate(self.names)}

    def load_tensor(self, i: int, value: np.ndarray) -> None:
        v = np.ascontiguousarray(value, dtype=np.float32).reshape(self.shapes[i])
        check(self.lib.gpt2_load_tensor(self.h, i, v.ctypes.data), "gpt2_load_tensor")

    def losses(self, B: int, T: int) -> np.ndarray:
        out = np.empty((B, T), dtype=np.float32)
        check(self.lib.gpt2_copy_losses(self.h, out.ctypes.data), "gpt2_copy_losses")
        return out

    def num_params(self) -> int:
        return int(self.lib.gpt2_num_params(self.h))

    def flat_params(self) -> int:
        """Length of the flat parameter layout (tensors on 64-element boundaries)."""
        return int(self.lib.gpt2_flat_params(self.h))

    def launch_count(self) -> int:
        return int(self.lib.gpt2_launch_count(self.h))

    def family_stats(self) -> dict:
        out = {}
        for f, name in enumerate(FAMILIES):
            calls, launches, work = c_int64(), c_int64(), c_double()
            check(self.lib.gpt2_family_stats(self.h, f, ctypes.byref(calls), ctypes.byref(launches),
                                             ctypes.byref(work)), "gpt2_family_stats")
            out[name] = {"calls": calls.value, "launches": launches.value, "work": work.value}
        return out

    def set_timing(self, enable: bool) -> None:
        check(self.lib.gpt2_set_timing(self.h, int(enable)), "gpt2_set_timing")

    def family_times_ms(self) -> dict:
        out = {}
        for f, name in enumerate(FAMILIES):
            ms = c_double()
            check(self.lib.gpt2_family_time(self.h, f, ctypes.byref(ms)), "gpt2_family_time")
            out[name] = ms.value
        return out

    def reset_stats(self) -> None:
        check(self.lib.gpt2_reset_stats(self.h), "gpt2_reset_stats")


# ---------------------------------------------------------------- per-kernel entry points (gpt2_ops.h)

def _p(t):
    return None if t is None else t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_of(t) -> int:
    import torch
    return MODE_BF16 if t.dtype == torch.bfloat16 else MODE_FP32


def _scratch(nbytes: int):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def gpt2_op_encoder_forward(x0, tokens, wte, wpe, V, status=None, stream=None):
    B, T = tokens.shape
    C = wte.shape[1]
    check(load_library().gpt2_op_encoder_forward(_dtype_of(x0), _p(x0), _p(tokens), _p(wte), _p(wpe), B, T, C, V,
                                                 _p(status), _s(stream)), "gpt2_op_encoder_forward")


def gpt2_op_encoder_backward(dwte, dwpe, dx0, tokens, stream=None):
    B, T = tokens.shape
    C = dwte.shape[1]
    lib = load_library()
    n = lib.gpt2_op_encoder_backward_scratch(B, T, C)
    sc = _scratch(n)
    check(lib.gpt2_op_encoder_backward(_dtype_of(dx0), _p(dwte), _p(dwpe), _p(dx0), _p(tokens), B, T, C,
                                       dwte.shape[0], _p(sc), sc.numel(), _s(stream)), "gpt2_op_encoder_backward")
    return sc


def gpt2_op_layernorm_forward(y, mean, rstd, x, gamma, beta, stream=None):
    N, C = x.shape
    check(load_library().gpt2_op_layernorm_forward(_dtype_of(x), _p(y), _p(mean), _p(rstd), _p(x), _p(gamma),
                                                   _p(beta), N, C, _s(stream)), "gpt2_op_layernorm_forward")


def gpt2_op_layernorm_backward(dx, dgamma, dbeta, dy, x, gamma, mean, rstd, stream=None):
    N, C = x.shape
    lib = load_library()
    sc = _scratch(lib.gpt2_op_layernorm_backward_scratch(N, C))
    check(lib.gpt2_op_layernorm_backward(_dtype_of(x), _p(dx), _p(dgamma), _p(dbeta), _p(dy), _p(x), _p(gamma),
                                         _p(mean), _p(rstd), N, C, _p(sc), sc.numel(), _s(stream)),
          "gpt2_op_layernorm_backward")
    return sc


def gpt2_op_residual_layernorm_forward(y, mean, rstd, xsum, x, r, gamma, beta, stream=None):
    N, C = x.shape
    check(load_library().gpt2_op_residual_layernorm_forward(_dtype_of(x), _p(y), _p(mean), _p(rstd), _p(xsum), _p(x),
                                                            _p(r), _p(gamma), _p(beta), N, C, _s(stream)),
          "gpt2_op_residual_layernorm_forward")


def gpt2_op_layernorm_backward_residual(dres, accumulate, dgamma, dbeta, dres_colsum, dy, x, gamma, mean, rstd,
                                        stream=None):
    N, C = x.shape
    lib = load_library()
    sc = _scratch(lib.gpt2_op_layernorm_backward_scratch(N, C))
    check(lib.gpt2_op_layernorm_backward_residual(_dtype_of(x), _p(dres), int(accumulate), _p(dgamma), _p(dbeta),
                                                  _p(dres_colsum), _p(dy), _p(x), _p(gamma), _p(mean), _p(rstd), N,
                                                  C, _p(sc), sc.numel(), _s(stream)),
          "gpt2_op_layernorm_backward_residual")
    return sc


def gpt2_op_matmul(D, A, a_mn, B, b_mn, M, N, K, bias=None, status=None, stream=None):
    import torch
    lib = load_library()
    dt = _dtype_of(A)
    d_fp32 = int(D.dtype == torch.float32)
    sc = _scratch(lib.gpt2_op_matmul_scratch(dt, M, N, K, d_fp32))
    check(lib.gpt2_op_matmul(dt, _p(D), d_fp32, _p(A), int(a_mn), _p(B), int(b_mn), _p(bias), M, N, K, _p(sc),
                             sc.numel(), _p(status), _s(stream)), "gpt2_op_matmul")
    return sc


def gpt2_lr_cosine(t: int, warmup: int, total: int, lr_max: float, lr_min: float) -> float:
    return float(load_library().gpt2_lr_cosine(int(t), int(warmup), int(total), float(lr_max), float(lr_min)))


def gpt2_op_quantize_fp8(q, scales, x, fmt=FP8_E4M3, stream=None):
    """q (uint8 [n]) = FP8 codes (format fmt) of x (bf16) scaled per tensor;
    scales (float32 [2]) = fmax/amax, amax/fmax (fmax 448 for e4m3, 57344 for e5m2)."""
    lib = load_library()
    sc = _scratch(lib.gpt2_op_quantize_fp8_scratch())
    check(lib.gpt2_op_quantize_fp8(_p(q), _p(scales), _p(x), x.numel(), int(fmt), _p(sc), sc.numel(), _s(stream)),
          "gpt2_op_quantize_fp8")


def gpt2_op_matmul_fp8(D, A, a_scales, B, b_scales, bias=None, a_fmt=FP8_E4M3, b_fmt=FP8_E4M3, status=None,
                       stream=None):
    """D (bf16 [M,N]) = (A B^T) a_scales[1] b_scales[1] (+ bias); A [M,K], B [N,K] FP8 codes (uint8) in
    formats a_fmt and b_fmt."""
    M, K = A.shape
    N = B.shape[0]
    check(load_library().gpt2_op_matmul_fp8(_p(D), _p(A), int(a_fmt), _p(a_scales), _p(B), int(b_fmt),
                                            _p(b_scales), _p(bias), M, N, K, _p(status), _s(stream)),
          "gpt2_op_matmul_fp8")


def gpt2_op_quantize_fp8_transpose(qt, scales, x, q=None, fmt=FP8_E4M3, stream=None):
    """qt (uint8 [C, R]) = the FP8 codes of x (bf16 [R, C]) under scales (from
    gpt2_op_quantize_fp8 of the same x), transposed; q (uint8 [R, C], optional)
    the same codes untransposed."""
    R, C = x.shape
    check(load_library().gpt2_op_quantize_fp8_transpose(_p(qt), _p(q), _p(scales), _p(x), R, C, int(fmt),
                                                        _s(stream)), "gpt2_op_quantize_fp8_transpose")


def gpt2_op_matmul_fp8_ex(epi, D, A, a_scales, B, b_scales, D2=None, aux=None, bias=None, accumulate=False,
                          a_fmt=FP8_E4M3, b_fmt=FP8_E4M3, status=None, stream=None):
    """The general FP8 product (gpt2_op_matmul_fp8_ex): epi 0 plain (D bf16 or
    fp32, accumulate into fp32 D), 1 the GELU forward (D = gelu'(u), D2 =
    gelu(u)), 2 the GELU backward (D = bf16(A B^T scales) * aux)."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    d_fp32 = int(D.dtype == torch.float32)
    lib = load_library()
    sc = _scratch(lib.gpt2_op_matmul_fp8_scratch(M, N, K, d_fp32, int(accumulate)))
    check(lib.gpt2_op_matmul_fp8_ex(int(epi), _p(D), _p(D2), _p(aux), d_fp32, int(accumulate), _p(A), int(a_fmt),
                                    _p(a_scales), _p(B), int(b_fmt), _p(b_scales), _p(bias), M, N, K, _p(sc),
                                    sc.numel(), _p(status), _s(stream)), "gpt2_op_matmul_fp8_ex")
    return sc


def gpt2_op_matmul_gelu(dgelu, out, A, W, bias=None, status=None, stream=None):
    """u = A W^T + bias; out = gelu(u), dgelu = gelu'(u); A [M, K], W [N, K]."""
    M, K = A.shape
    N = W.shape[0]
    check(load_library().gpt2_op_matmul_gelu(_dtype_of(A), _p(dgelu), _p(out), _p(A), _p(W), _p(bias), M, N, K,
                                             _p(status), _s(stream)), "gpt2_op_matmul_gelu")


def gpt2_op_matmul_gelu_backward(du, dY, W, dgelu, status=None, stream=None):
    """du = (dY W) * dgelu; dY [M, K], W [K, N], dgelu [M, N]."""
    M, K = dY.shape
    N = W.shape[1]
    check(load_library().gpt2_op_matmul_gelu_backward(_dtype_of(dY), _p(du), _p(dY), _p(W), _p(dgelu), M, N, K,
                                                      _p(status), _s(stream)), "gpt2_op_matmul_gelu_backward")


def gpt2_op_matmul_gelu_backward_bias(du, dbias, dY, W, dgelu, status=None, stream=None):
    """du = (dY W) * dgelu and dbias = column sums of du (fp32 [N])."""
    M, K = dY.shape
    N = W.shape[1]
    lib = load_library()
    sc = _scratch(lib.gpt2_op_matmul_gelu_backward_bias_scratch(M, N))
    check(lib.gpt2_op_matmul_gelu_backward_bias(_dtype_of(dY), _p(du), _p(dbias), _p(dY), _p(W), _p(dgelu), M, N,
                                                K, _p(sc), sc.numel(), _p(status), _s(stream)),
          "gpt2_op_matmul_gelu_backward_bias")
    return sc


def gpt2_op_attention_forward(o, lse, qkv, B, T, H, stream=None):
    C = qkv.shape[-1] // 3
    check(load_library().gpt2_op_attention_forward(_dtype_of(qkv), _p(o), _p(lse), _p(qkv), B, T, C, H,
                                                   _s(stream)), "gpt2_op_attention_forward")


def gpt2_op_attention_backward(dqkv, dout, qkv, o, lse, B, T, H, stream=None):
    C = qkv.shape[-1] // 3
    lib = load_library()
    sc = _scratch(lib.gpt2_op_attention_backward_scratch(B, T, H))
    check(lib.gpt2_op_attention_backward(_dtype_of(qkv), _p(dqkv), _p(dout), _p(qkv), _p(o), _p(lse), B, T, C, H,
                                         _p(sc), sc.numel(), _s(stream)), "gpt2_op_attention_backward")
    return sc


def gpt2_op_gelu_forward(g, u, stream=None):
    check(load_library().gpt2_op_gelu_forward(_dtype_of(u), _p(g), _p(u), u.numel(), _s(stream)),
          "gpt2_op_gelu_forward")


def gpt2_op_gelu_backward(du, u, dg, stream=None):
    check(load_library().gpt2_op_gelu_backward(_dtype_of(u), _p(du), _p(u), _p(dg), u.numel(), _s(stream)),
          "gpt2_op_gelu_backward")


def gpt2_op_residual_forward(out, a, b, stream=None):
    check(load_library().gpt2_op_residual_forward(_dtype_of(a), _p(out), _p(a), _p(b), a.numel(), _s(stream)),
          "gpt2_op_residual_forward")


def gpt2_op_residual_backward(dres, dbranch, stream=None):
    check(load_library().gpt2_op_residual_backward(_dtype_of(dres), _p(dres), _p(dbranch), dres.numel(),
                                                   _s(stream)), "gpt2_op_residual_backward")


def gpt2_op_bias_backward(dbias, dy, stream=None):
    N, C = dy.shape
    lib = load_library()
    sc = _scratch(lib.gpt2_op_bias_backward_scratch(N, C))
    check(lib.gpt2_op_bias_backward(_dtype_of(dy), _p(dbias), _p(dy), N, C, _p(sc), sc.numel(), _s(stream)),
          "gpt2_op_bias_backward")
    return sc


def gpt2_op_bias_backward_noalloc(dbias, dy, stream=None):
    """Bias gradient with the library's fixed internal scratch (no caller scratch)."""
    N, C = dy.shape
    check(load_library().gpt2_op_bias_backward_noalloc(_dtype_of(dy), _p(dbias), _p(dy), N, C, _s(stream)),
          "gpt2_op_bias_backward_noalloc")


def gpt2_op_classifier(logits, losses, targets, V, dloss, status=None, stream=None):
    N, Vp = logits.shape
    check(load_library().gpt2_op_classifier(_dtype_of(logits), _p(logits), _p(losses), _p(targets), N, V, Vp,
                                            dloss, _p(status), _s(stream)), "gpt2_op_classifier")


def gpt2_op_mean_loss(out, losses, stream=None):
    check(load_library().gpt2_op_mean_loss(_p(out), _p(losses), losses.numel(), _s(stream)), "gpt2_op_mean_loss")


def gpt2_op_adamw(master, param_bf16, grad, m, v, lr, beta1, beta2, eps, weight_decay, t, stream=None):
    check(load_library().gpt2_op_adamw(_p(master), _p(param_bf16), _p(grad), _p(m), _p(v), master.numel(), lr,
                                       beta1, beta2, eps, weight_decay, t, _s(stream)), "gpt2_op_adamw")
