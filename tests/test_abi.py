"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/llama_layer.h declares, and rejects bad arguments on
the host before touching the device."""

import ctypes
import os
import re

import pytest

from llama_decoder_layer_gb300 import binding as lb
from llama_decoder_layer_gb300 import build as lbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "llama_layer.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("typedef",)))


@pytest.fixture(scope="module")
def lib():
    lbuild.build()
    return lb.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("llama_layer_forward", "llama_stack_forward", "kv_cache_write", "llama_workspace_size",
                     "llama_status_string", "llama_get_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in llama_layer.h but not exported"
    # and the binding knows every one of them
    assert set(names) == set(lb.SIGNATURES), set(names) ^ set(lb.SIGNATURES)


def test_status_strings(lib):
    for st in range(0, 8):
        s = lb.status_string(st)
        assert s and "unknown" not in s
    assert "unknown" in lb.status_string(99)


def test_host_argument_checks_without_a_gpu(lib):
    L = lib
    # null config / weights / batch
    assert L.llama_layer_forward(None, None, None, None, None, None, None, None, None, 0, None) == lb.LLAMA_ERR_ARG
    cfg = lb.LayerConfig(512, 8, 2, 64, 1376, 1e-5, 1e4)
    c = cfg.c()
    assert L.llama_layer_forward(ctypes.byref(c), None, None, None, None, None, None, None, None, 0,
                                 None) == lb.LLAMA_ERR_ARG
    # unsupported activation (the MLP accepts silu only)
    bad = lb.LayerConfig(512, 8, 2, 64, 1376, 1e-5, 1e4, hidden_act="gelu").c()
    assert L.llama_paged_attention(ctypes.byref(bad), None, None, None, None, None, None, 0,
                                   None) == lb.LLAMA_ERR_ARG
    # n_heads not a multiple of n_kv_heads
    bad = lb.LayerConfig(512, 8, 3, 64, 1376, 1e-5, 1e4).c()
    assert L.llama_paged_attention(ctypes.byref(bad), None, None, None, None, None, None, 0,
                                   None) == lb.LLAMA_ERR_ARG
    # head_dim outside {64, 128}
    bad = lb.LayerConfig(512, 8, 2, 96, 1376, 1e-5, 1e4).c()
    assert L.llama_paged_attention(ctypes.byref(bad), None, None, None, None, None, None, 0,
                                   None) == lb.LLAMA_ERR_UNSUPPORTED
    # GQA group above 16
    bad = lb.LayerConfig(4096, 32, 1, 128, 1376, 1e-5, 1e4).c()
    assert L.llama_paged_attention(ctypes.byref(bad), None, None, None, None, None, None, 0,
                                   None) == lb.LLAMA_ERR_UNSUPPORTED
    # the stack needs at least one layer
    assert L.llama_stack_forward(ctypes.byref(c), 0, None, None, None, 0, None, None, None, None, None, None, None,
                                 None, None, None, 0, None) == lb.LLAMA_ERR_ARG
    # cache write: bad sizes
    assert L.kv_cache_write(None, None, None, 4, 0, 128, 16, 10, None, None, None) == lb.LLAMA_ERR_ARG
    assert L.kv_cache_write(None, None, None, 4, 8, 100, 16, 10, None, None, None) == lb.LLAMA_ERR_ARG
    # empty problems are valid no-ops
    assert L.kv_cache_write(None, None, None, 0, 8, 128, 16, 10, None, None, None) == lb.LLAMA_OK
    assert L.llama_linear(None, None, 0, 256, 256, None, 0, None, 0, None) == lb.LLAMA_OK
    assert L.llama_linear(None, None, 4, 250, 256, None, 0, None, 0, None) == lb.LLAMA_ERR_ARG  # null pointers first
    # norm: H must be a multiple of 8 within 16384
    assert L.llama_fused_add_rmsnorm(None, None, None, None, None, 4, 100, 1e-5, None) == lb.LLAMA_ERR_ARG
    # folded norms: both norm weights NULL or neither (fake aligned addresses; rejected before any launch)
    fake = 256
    half = lb.LlamaLayerWeights(None, fake, fake, fake, fake, fake)
    assert L.llama_layer_forward(ctypes.byref(c), ctypes.byref(half), None, None, None, None, None, None, None, 0,
                                 None) == lb.LLAMA_ERR_ARG
    # fold: null pointers, then columns that are not a multiple of 8
    assert L.llama_fold_norm_weights(None, None, 4, 64, None, None) == lb.LLAMA_ERR_ARG
    assert L.llama_fold_norm_weights(fake, fake, 4, 60, fake, None) == lb.LLAMA_ERR_UNSUPPORTED



def test_launch_counter_counts_only_accepted_launches(lib):
    # a call rejected on the host launches nothing; the counter is monotonic
    before = lb.launch_count()
    assert lib.llama_linear(None, None, 4, 250, 256, None, 0, None, 0, None) == lb.LLAMA_ERR_ARG
    assert lb.launch_count() == before


def test_gate_up_timer_and_schedule_argument_checks(lib):
    # both are rejected on the host before any CUDA call
    assert lib.llama_gate_up_timer_start(0) == lb.LLAMA_ERR_ARG
    assert lib.llama_gate_up_timer_start(-5) == lb.LLAMA_ERR_ARG
    ms, n = ctypes.c_float(0.0), ctypes.c_int(0)
    assert lib.llama_gate_up_timer_stop(ctypes.byref(ms), ctypes.byref(n)) == lb.LLAMA_ERR_ARG  # not running
    assert lib.llama_set_gemm_schedule(7) == lb.LLAMA_ERR_ARG
    assert lib.llama_set_gemm_schedule(-2) == lb.LLAMA_ERR_ARG
    assert lib.llama_set_gemm_schedule(-1) == lb.LLAMA_OK


def test_sampler_host_argument_checks(lib):
    fake = ctypes.c_void_p(256)
    assert lib.llama_sample(None, 0, 10, None, None, None, None, None, None, None) == lb.LLAMA_OK  # no rows
    assert lib.llama_sample(fake, -1, 10, fake, fake, fake, fake, fake, None, None) == lb.LLAMA_ERR_ARG
    assert lib.llama_sample(fake, 4, 0, fake, fake, fake, fake, fake, None, None) == lb.LLAMA_ERR_ARG
    assert lib.llama_sample(fake, 4, 10, fake, None, fake, fake, fake, None, None) == lb.LLAMA_ERR_ARG
    assert lib.llama_sample(fake, 4, 10, fake, fake, fake, None, fake, None, None) == lb.LLAMA_ERR_ARG


def test_moe_host_argument_checks(lib):
    # rejected on the host, before anything touches the (fake) device pointers
    fake = ctypes.c_void_p(256)
    MC = lb.LlamaMoeConfig
    good = MC(2048, 128, 8, 768)
    assert lib.llama_moe_workspace_size(ctypes.byref(good), 64) > 0
    assert lib.llama_moe_workspace_size(None, 64) == 0
    assert lib.llama_moe_workspace_size(ctypes.byref(MC(2048, 8, 9, 768)), 64) == 0  # top_k > experts
    assert lib.llama_moe_workspace_size(ctypes.byref(good), -1) == 0
    args = (fake, fake, fake, fake, fake, None, None, fake, 1 << 30, None)
    assert lib.llama_moe_forward(None, fake, 4, *args[1:]) == lb.LLAMA_ERR_ARG
    assert lib.llama_moe_forward(ctypes.byref(MC(2048, 128, 0, 768)), fake, 4, *args[1:]) == lb.LLAMA_ERR_ARG
    assert lib.llama_moe_forward(ctypes.byref(MC(2044, 128, 8, 768)), fake, 4, *args[1:]) == lb.LLAMA_ERR_UNSUPPORTED
    assert lib.llama_moe_forward(ctypes.byref(MC(2048, 600, 8, 768)), fake, 4, *args[1:]) == lb.LLAMA_ERR_UNSUPPORTED
    assert lib.llama_moe_forward(ctypes.byref(good), fake, 0, *args[1:]) == lb.LLAMA_OK  # no tokens
    assert lib.llama_moe_forward(ctypes.byref(good), fake, -1, *args[1:]) == lb.LLAMA_ERR_ARG
    assert lib.llama_moe_forward(ctypes.byref(good), None, 4, *args[1:]) == lb.LLAMA_ERR_ARG
    # too small a workspace
    assert lib.llama_moe_forward(ctypes.byref(good), fake, 4, fake, fake, fake, fake, None, None, fake, 16,
                                 None) == lb.LLAMA_ERR_WORKSPACE


def test_moe_layer_host_argument_checks(lib):
    fake = 256
    cfg = lb.LayerConfig(2048, 32, 4, 128, 6144, 1e-6, 1e7).c()
    good = lb.LlamaMoeConfig(2048, 128, 8, 768)
    assert lib.llama_moe_layer_workspace_size(ctypes.byref(cfg), ctypes.byref(good), 64, 64, 4096) > 0
    # the block's hidden size must be the layer's
    other = lb.LlamaMoeConfig(1024, 128, 8, 768)
    assert lib.llama_moe_layer_workspace_size(ctypes.byref(cfg), ctypes.byref(other), 64, 64, 4096) == 0
    w = lb.LlamaMoeLayerWeights(fake, fake, fake, fake, fake, fake, fake)
    assert lib.llama_moe_layer_forward(ctypes.byref(cfg), ctypes.byref(other), ctypes.byref(w), None, None, None,
                                       None, None, None, None, None, 0, None) == lb.LLAMA_ERR_ARG
    # a missing expert weight
    w_bad = lb.LlamaMoeLayerWeights(fake, fake, fake, fake, fake, None, fake)
    assert lib.llama_moe_layer_forward(ctypes.byref(cfg), ctypes.byref(good), ctypes.byref(w_bad), None, None, None,
                                       None, None, None, None, None, 0, None) == lb.LLAMA_ERR_ARG
    # the MoE layer needs its norm weights (no folded form)
    w_fold = lb.LlamaMoeLayerWeights(None, fake, fake, None, fake, fake, fake)
    assert lib.llama_moe_layer_forward(ctypes.byref(cfg), ctypes.byref(good), ctypes.byref(w_fold), None, None, None,
                                       None, None, None, None, None, 0, None) == lb.LLAMA_ERR_ARG
