"""ctypes binding of include/gpt2.h: loads the in-tree libgpt2_b300.so and declares
every entry point.  Argument marshalling only; there is no other code path.

Importing this module raises if the library has not been built (run
``python -m gpt_train_step_arena_b300.build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes as ct
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpt2_b300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                      "(python -m gpt_train_step_arena_b300.build)")

lib = ct.CDLL(LIB_PATH)

P, I, U64, SZ, F = ct.c_void_p, ct.c_int, ct.c_uint64, ct.c_size_t, ct.c_float

# name: (restype, argtypes) — mirrors include/gpt2.h
SIGNATURES = {
    "gpt2_build_ex": (P, [I, I, I, I, I, I, ct.POINTER(I)]),
    "gpt2_build_norm": (P, [I, I, I, I, I, I, I, ct.POINTER(I)]),
    "gpt2_build": (P, [I, I, I, I, I]),
    "gpt2_free": (None, [P]),
    "gpt2_num_params": (SZ, [P]),
    "gpt2_padded_vocab": (I, [P]),
    "gpt2_init_params": (I, [P, U64]),
    "gpt2_set_params": (I, [P, P, SZ]),
    "gpt2_get_params": (I, [P, P, SZ]),
    "gpt2_get_grads": (I, [P, P, SZ]),
    "gpt2_get_opt_state": (I, [P, P, P, SZ]),
    "gpt2_forward": (F, [P, P, P, I, I]),
    "gpt2_forward_async": (I, [P, P, P, I, I, I]),
    "gpt2_read_loss": (I, [P, ct.POINTER(F)]),
    "gpt2_backward": (I, [P]),
    "gpt2_zero_grad": (I, [P]),
    "gpt2_update": (I, [P, F, F, F, F, F, I]),
    "gpt2_get_losses": (I, [P, P, SZ]),
    "gpt2_get_logits": (I, [P, P, SZ]),
    "gpt2_generate": (I, [P, P, I, I, I, F, P, P]),
    "gpt2_get_gen_logits": (I, [P, P, SZ]),
    "gpt2_get_ids": (I, [P, P, P, SZ]),
    "gpt2_profile_enable": (I, [P, I]),
    "gpt2_profile_reset": (I, [P]),
    "gpt2_profile_read": (I, [P, I, ct.POINTER(ct.c_double), ct.POINTER(ct.c_double), ct.POINTER(U64)]),
    "gpt2_check_bounded_wait": (I, [P, ct.c_uint]),
    "gpt2_set_stream": (I, [P, P]),
    "gpt2_sync": (I, [P]),
    "gpt2_last_status": (I, [P]),
    "gpt2_last_error": (ct.c_char_p, [P]),
    "gpt2_last_build_error": (ct.c_char_p, []),
    "gpt2_kernel_launches": (U64, [P]),
    "gpt2_device_bytes": (SZ, [P]),
    # include/gpt2_ops.h
    "gpt2_op_last_error": (ct.c_char_p, []),
    "gpt2_op_bias_grad_workspace": (SZ, [I, I]),
    "gpt2_op_bias_grad": (I, [I, P, I, I, P, P, SZ, P]),
    "gpt2_op_bias_grad_noalloc": (I, [I, P, I, I, P, P]),
    "gpt2_op_bias_grad_noalloc_max_floats": (SZ, []),
    "gpt2_op_matmul": (I, [I, I, I, I, P, ct.c_longlong, I, P, ct.c_longlong, I, P, ct.c_longlong, I, P, P, SZ, P]),
    "gpt2_op_matmul_workspace": (SZ, [I, I, I, I, I, I]),
    "gpt2_op_matmul_ex": (I, [I, I, I, I, P, ct.c_longlong, I, P, ct.c_longlong, I, P, ct.c_longlong, P, P,
                              ct.c_longlong, P, ct.c_longlong, P, ct.c_longlong, I, P, SZ, P]),
    "gpt2_op_matmul_gelu_bwd_bias_grad_workspace": (SZ, [I, I]),
    "gpt2_op_matmul_gelu_bwd_bias_grad": (I, [I, I, I, P, ct.c_longlong, I, P, ct.c_longlong, I, P, ct.c_longlong,
                                              P, ct.c_longlong, P, P, SZ, P]),
    "gpt2_op_adamw": (I, [P, P, P, P, P, SZ, F, F, F, F, F, I, P]),
    "gpt2_op_attention_forward": (I, [I, P, P, P, I, I, I, I, P]),
    "gpt2_op_attention_backward": (I, [I, P, P, P, P, P, I, I, I, I, P, P]),
    "gpt2_op_layernorm_forward": (I, [I, P, P, P, P, P, P, I, I, P]),
    "gpt2_op_layernorm_backward_workspace": (SZ, [I]),
    "gpt2_op_layernorm_backward": (I, [I, P, P, P, P, P, P, P, P, I, I, P, SZ, P]),
    "gpt2_op_rmsnorm_forward": (I, [I, P, P, P, P, I, I, P]),
    "gpt2_op_rmsnorm_backward_workspace": (SZ, [I]),
    "gpt2_op_rmsnorm_backward": (I, [I, P, P, P, P, P, P, I, I, P, SZ, P]),
    "gpt2_op_softmax_xent": (I, [I, P, P, P, I, I, I, F, P, P]),
    "gpt2_op_encoder_forward": (I, [I, P, P, P, P, I, I, I, I, P, P]),
    "gpt2_op_encoder_backward_workspace": (SZ, [I, I, I]),
    "gpt2_op_encoder_backward": (I, [I, P, P, P, P, I, I, I, I, I, P, SZ, P]),
    "gpt2_op_gemm_force_tile_rows": (I, [I]),
    "gpt2_op_gemm_last_variant": (ct.c_char_p, []),
}

for _name, (_res, _args) in SIGNATURES.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

# enum values of include/gpt2.h
GPT2_OK, GPT2_ERR_ARG, GPT2_ERR_OOM, GPT2_ERR_CUDA = 0, -1, -2, -3
GPT2_ERR_TOKEN, GPT2_ERR_SHAPE, GPT2_ERR_STATE, GPT2_ERR_NONFINITE, GPT2_ERR_TIMEOUT = -4, -5, -6, -7, -8
GPT2_FP32, GPT2_TF32, GPT2_BF16 = 0, 1, 2
GPT2_LAYERNORM, GPT2_RMSNORM = 0, 1
GPT2_DT_F32, GPT2_DT_BF16, GPT2_DT_TF32 = 0, 1, 2
GPT2_HOST, GPT2_DEVICE = 0, 1
GPT2_EPI_STORE, GPT2_EPI_GELU, GPT2_EPI_GELU_BWD = 0, 1, 2
KERNEL_CLASSES = ["gemm", "attn_fwd", "attn_bwd", "layernorm", "xent", "adamw", "encoder", "bias_grad"]

STATUS_NAMES = {0: "GPT2_OK", -1: "GPT2_ERR_ARG", -2: "GPT2_ERR_OOM", -3: "GPT2_ERR_CUDA",
                -4: "GPT2_ERR_TOKEN", -5: "GPT2_ERR_SHAPE", -6: "GPT2_ERR_STATE",
                -7: "GPT2_ERR_NONFINITE", -8: "GPT2_ERR_TIMEOUT"}
