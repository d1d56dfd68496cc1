"""Python binding of the C ABI in ``include/llama_layer.h``.

Argument marshalling only: torch tensors become device pointers, Python ints
become C ints, and a non-zero status raises :class:`LlamaError`.  Every step
of the computation runs in the CUDA library; if the library is missing this
module raises instead of computing anything itself.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import build as _build

LLAMA_OK = 0
LLAMA_ERR_ARG = 1
LLAMA_ERR_UNSUPPORTED = 2
LLAMA_ERR_CUDA = 3
LLAMA_ERR_WORKSPACE = 4
LLAMA_ERR_DEVICE_GUARD = 5
LLAMA_ERR_TIMEOUT = 6
LLAMA_ERR_SCRATCH_LIMIT = 7


class LlamaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class LlamaLayerConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("intermediate", ctypes.c_int), ("block_size", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("rope_scaling", ctypes.c_int),
                ("rs_factor", ctypes.c_float), ("rs_low_freq_factor", ctypes.c_float),
                ("rs_high_freq_factor", ctypes.c_float), ("rs_original_max_pos", ctypes.c_int),
                ("hidden_act", ctypes.c_int)]


class LlamaLayerWeights(ctypes.Structure):
    _fields_ = [("ln1_w", ctypes.c_void_p), ("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("ln2_w", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


class LlamaMoeConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("num_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("moe_intermediate", ctypes.c_int)]


class LlamaMoeLayerWeights(ctypes.Structure):
    _fields_ = [("ln1_w", ctypes.c_void_p), ("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("ln2_w", ctypes.c_void_p), ("w_router", ctypes.c_void_p), ("w13", ctypes.c_void_p),
                ("w2", ctypes.c_void_p)]


class LlamaBatch(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int), ("num_seqs", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("max_query_len", ctypes.c_int), ("max_seq_len", ctypes.c_int),
                ("positions", ctypes.c_void_p), ("query_start_loc", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("slot_mapping", ctypes.c_void_p)]


# every entry point of include/llama_layer.h with its C signature
_VP, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_P_CFG, _P_W, _P_B = ctypes.POINTER(LlamaLayerConfig), ctypes.POINTER(LlamaLayerWeights), ctypes.POINTER(LlamaBatch)
SIGNATURES = {
    "llama_workspace_size": (_SZ, [_P_CFG, _I, _I, _I, _I]),
    "llama_layer_forward": (_I, [_P_CFG, _P_W, _P_B, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "llama_stack_forward": (_I, [_P_CFG, _I, _P_W, _VP, _VP, _I, _VP, _VP, _P_B, _VP, _VP, _VP, _VP, _VP, _VP,
                                 _VP, _SZ, _VP]),
    "kv_cache_write": (_I, [_VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _VP]),
    "llama_linear": (_I, [_VP, _VP, _I, _I, _I, _VP, _I, _VP, _SZ, _VP]),
    "llama_linear_workspace_size": (_SZ, []),
    "llama_gate_up_silu": (_I, [_VP, _VP, _I, _I, _I, _VP, _VP, _SZ, _VP]),
    "llama_fused_add_rmsnorm": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _F, _VP]),
    "llama_paged_attention": (_I, [_P_CFG, _P_B, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "llama_paged_attention_noalloc": (_I, [_P_CFG, _P_B, _VP, _VP, _VP, _VP, _VP]),
    "llama_paged_attention_noalloc_limit": (_SZ, []),
    "llama_get_device_error": (_I, [_VP, ctypes.POINTER(ctypes.c_int)]),
    "llama_status_string": (ctypes.c_char_p, [_I]),
    "llama_num_sms": (_I, []),
    "llama_launch_count": (ctypes.c_uint64, []),
    "llama_set_gemm_schedule": (_I, [_I]),
    "llama_gate_up_timer_start": (_I, [_I]),
    "llama_gate_up_timer_stop": (_I, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]),
    "llama_sample": (_I, [_VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "llama_moe_workspace_size": (_SZ, [ctypes.POINTER(LlamaMoeConfig), _I]),
    "llama_moe_forward": (_I, [ctypes.POINTER(LlamaMoeConfig), _VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "llama_fold_norm_weights": (_I, [_VP, _VP, _I, _I, _VP, _VP]),
    "llama_selftest_wait_timeout": (_I, [_VP]),
    "llama_moe_layer_workspace_size": (_SZ, [_P_CFG, ctypes.POINTER(LlamaMoeConfig), _I, _I, _I]),
    "llama_moe_layer_forward": (_I, [_P_CFG, ctypes.POINTER(LlamaMoeConfig), ctypes.POINTER(LlamaMoeLayerWeights),
                                     _P_B, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
}

_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m llama_decoder_layer_gb300.build` "
                               "(there is no fallback implementation)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().llama_status_string(int(status)).decode()
    except Exception:
        return f"status {status}"


def _check(status: int, where: str) -> None:
    if status != LLAMA_OK:
        raise LlamaError(status, where)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class LayerConfig:
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    rms_eps: float
    rope_theta: float
    rope_scaling: Optional[dict] = None
    block_size: int = 16
    hidden_act: str = "silu"

    def c(self) -> LlamaLayerConfig:
        s = self.rope_scaling or {}
        return LlamaLayerConfig(
            self.hidden, self.n_heads, self.n_kv_heads, self.head_dim, self.intermediate, self.block_size,
            self.rms_eps, self.rope_theta, 1 if self.rope_scaling else 0, float(s.get("factor", 1.0)),
            float(s.get("low_freq_factor", 1.0)), float(s.get("high_freq_factor", 1.0)),
            int(s.get("original_max_position_embeddings", 0)), 0 if self.hidden_act == "silu" else 1)

    @staticmethod
    def from_spec(spec) -> "LayerConfig":
        return LayerConfig(spec.hidden, spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.intermediate,
                           spec.rms_eps, spec.rope_theta, spec.rope_scaling, spec.block_size)


def make_weights(w: dict) -> LlamaLayerWeights:
    return LlamaLayerWeights(_ptr(w["ln1"]), _ptr(w["w_qkv"]), _ptr(w["w_o"]), _ptr(w["ln2"]),
                             _ptr(w["w_gate_up"]), _ptr(w["w_down"]))


@dataclass
class Batch:
    """Device metadata of one flat batch plus the host bounds the launches need."""

    positions: torch.Tensor
    query_start_loc: torch.Tensor
    seq_lens: torch.Tensor
    block_table: torch.Tensor
    num_blocks: int
    max_query_len: int
    max_seq_len: int
    slot_mapping: Optional[torch.Tensor] = None

    @staticmethod
    def from_layout(bl, slot_mapping=None) -> "Batch":
        seq_lens = [c + q for c, q in zip(bl.ctx_lens, bl.q_lens)]
        return Batch(bl.positions, bl.query_start_loc, bl.seq_lens, bl.block_table, bl.num_blocks,
                     max(bl.q_lens), max(seq_lens), slot_mapping)

    def c(self) -> LlamaBatch:
        T = int(self.positions.numel())
        B = int(self.seq_lens.numel())
        return LlamaBatch(T, B, int(self.block_table.shape[1]), int(self.num_blocks), int(self.max_query_len),
                          int(self.max_seq_len), _ptr(self.positions), _ptr(self.query_start_loc),
                          _ptr(self.seq_lens), _ptr(self.block_table), _ptr(self.slot_mapping))


def workspace_size(cfg: LayerConfig, max_tokens: int, max_seqs: int, max_seq_len: int, vocab: int = 0) -> int:
    c = cfg.c()
    n = lib().llama_workspace_size(ctypes.byref(c), max_tokens, max_seqs, max_seq_len, vocab)
    if n == 0:
        raise LlamaError(LLAMA_ERR_ARG, "llama_workspace_size")
    return int(n)


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def layer_forward(cfg: LayerConfig, weights: dict, batch: Batch, hidden: torch.Tensor,
                  residual_in: Optional[torch.Tensor], residual_out: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    c, w, b = cfg.c(), make_weights(weights), batch.c()
    st = lib().llama_layer_forward(ctypes.byref(c), ctypes.byref(w), ctypes.byref(b), _ptr(hidden),
                                   _ptr(residual_in), _ptr(residual_out), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "llama_layer_forward")


def stack_forward(cfg: LayerConfig, layers: Sequence[dict], final_norm: torch.Tensor, lm_head: torch.Tensor,
                  batch: Batch, hidden: torch.Tensor, residual: torch.Tensor, k_caches: Sequence[torch.Tensor],
                  v_caches: Sequence[torch.Tensor], out_tokens: torch.Tensor, workspace: torch.Tensor,
                  embed: Optional[torch.Tensor] = None, input_ids: Optional[torch.Tensor] = None,
                  out_logits: Optional[torch.Tensor] = None, stream=None) -> None:
    n = len(layers)
    c, b = cfg.c(), batch.c()
    ws_arr = (LlamaLayerWeights * n)(*[make_weights(w) for w in layers])
    kc = (ctypes.c_void_p * n)(*[_ptr(t) for t in k_caches])
    vc = (ctypes.c_void_p * n)(*[_ptr(t) for t in v_caches])
    st = lib().llama_stack_forward(ctypes.byref(c), n, ws_arr, _ptr(final_norm), _ptr(lm_head),
                                   int(lm_head.shape[0]), _ptr(embed), _ptr(input_ids), ctypes.byref(b),
                                   _ptr(hidden), _ptr(residual), kc, vc, _ptr(out_tokens), _ptr(out_logits),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "llama_stack_forward")


def kv_cache_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, block_size: int = 16, stream=None) -> None:
    T, nkv, d = k.shape
    st = lib().kv_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, nkv, d, block_size, int(k_cache.shape[0]),
                              _ptr(k_cache), _ptr(v_cache), _stream(stream))
    _check(st, "kv_cache_write")


def linear(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    M, K = x.shape
    N = w.shape[0]
    st = lib().llama_linear(_ptr(x), _ptr(w), M, N, K, _ptr(out), 1 if out.dtype == torch.float32 else 0,
                            _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "llama_linear")


def gate_up_silu(x: torch.Tensor, w_gate_up: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                 stream=None) -> None:
    M, K = x.shape
    I = w_gate_up.shape[0] // 2
    st = lib().llama_gate_up_silu(_ptr(x), _ptr(w_gate_up), M, I, K, _ptr(out), _ptr(workspace), workspace.numel(),
                                  _stream(stream))
    _check(st, "llama_gate_up_silu")


def linear_workspace_size() -> int:
    return int(lib().llama_linear_workspace_size())


def fused_add_rmsnorm(x, residual_in, residual_out, h, gamma, eps: float, stream=None) -> None:
    rows, H = x.shape
    st = lib().llama_fused_add_rmsnorm(_ptr(x), _ptr(residual_in), _ptr(residual_out), _ptr(h), _ptr(gamma), rows, H,
                                       float(eps), _stream(stream))
    _check(st, "llama_fused_add_rmsnorm")


def paged_attention(cfg: LayerConfig, batch: Batch, q, k_cache, v_cache, out, workspace, stream=None) -> None:
    c, b = cfg.c(), batch.c()
    st = lib().llama_paged_attention(ctypes.byref(c), ctypes.byref(b), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "llama_paged_attention")


def paged_attention_noalloc(cfg: LayerConfig, batch: Batch, q, k_cache, v_cache, out, stream=None) -> None:
    """Paged attention with the library's fixed scratch array instead of a
    workspace, for callers that cannot allocate device memory."""
    c, b = cfg.c(), batch.c()
    st = lib().llama_paged_attention_noalloc(ctypes.byref(c), ctypes.byref(b), _ptr(q), _ptr(k_cache),
                                             _ptr(v_cache), _ptr(out), _stream(stream))
    _check(st, "llama_paged_attention_noalloc")


def set_gemm_schedule(schedule: int) -> None:
    """Process-wide GEMM schedule: -1 automatic, 0 single-SM tiles, 1 stream-K,
    2 cluster split-K, 3 SM-pair tiles."""
    _check(lib().llama_set_gemm_schedule(int(schedule)), "llama_set_gemm_schedule")


def gate_up_timer_start(max_launches: int) -> None:
    """Time every gate_up GEMM launch of the layer and stack calls from now on."""
    _check(lib().llama_gate_up_timer_start(int(max_launches)), "llama_gate_up_timer_start")


def gate_up_timer_stop():
    """(total ms, launches) of the gate_up launches timed since the start."""
    ms, n = ctypes.c_float(0.0), ctypes.c_int(0)
    _check(lib().llama_gate_up_timer_stop(ctypes.byref(ms), ctypes.byref(n)), "llama_gate_up_timer_stop")
    return float(ms.value), int(n.value)


def get_device_error(stream=None):
    """(status, detail) of the device error word; synchronises and clears it."""
    d = ctypes.c_int(0)
    st = lib().llama_get_device_error(_stream(stream), ctypes.byref(d))
    return st, d.value


def num_sms() -> int:
    return int(lib().llama_num_sms())


def sample(logits: torch.Tensor, temperature: torch.Tensor, top_k: torch.Tensor, top_p: torch.Tensor,
           uniform: torch.Tensor, out_tokens: torch.Tensor, out_logprobs: Optional[torch.Tensor] = None,
           stream=None) -> None:
    """Temperature / top-k / top-p sampling of fp32 logits [rows, vocab] with
    the caller's uniforms (one per row); see llama_sample in the header."""
    rows, vocab = logits.shape
    st = lib().llama_sample(_ptr(logits), rows, vocab, _ptr(temperature), _ptr(top_k), _ptr(top_p), _ptr(uniform),
                            _ptr(out_tokens), _ptr(out_logprobs), _stream(stream))
    _check(st, "llama_sample")


def moe_workspace_size(hidden: int, num_experts: int, top_k: int, moe_intermediate: int, max_tokens: int) -> int:
    c = LlamaMoeConfig(hidden, num_experts, top_k, moe_intermediate)
    return int(lib().llama_moe_workspace_size(ctypes.byref(c), max_tokens))


def moe_forward(h: torch.Tensor, w_router: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, top_k: int,
                out: torch.Tensor, workspace: torch.Tensor, out_ids: Optional[torch.Tensor] = None,
                out_weights: Optional[torch.Tensor] = None, stream=None) -> None:
    """The sparse MoE block over h [T, H]: w_router [E, H], w13 [E, 2I, H],
    w2 [E, H, I]; see llama_moe_forward in the header."""
    E, H = w_router.shape
    c = LlamaMoeConfig(H, E, top_k, int(w2.shape[2]))
    st = lib().llama_moe_forward(ctypes.byref(c), _ptr(h), int(h.shape[0]), _ptr(w_router), _ptr(w13), _ptr(w2),
                                 _ptr(out), _ptr(out_ids), _ptr(out_weights), _ptr(workspace), workspace.numel(),
                                 _stream(stream))
    _check(st, "llama_moe_forward")


def moe_layer_workspace_size(cfg: LayerConfig, num_experts: int, top_k: int, moe_intermediate: int,
                             max_tokens: int, max_seqs: int, max_seq_len: int) -> int:
    c = cfg.c()
    m = LlamaMoeConfig(c.hidden, num_experts, top_k, moe_intermediate)
    n = lib().llama_moe_layer_workspace_size(ctypes.byref(c), ctypes.byref(m), max_tokens, max_seqs, max_seq_len)
    if n == 0:
        raise LlamaError(LLAMA_ERR_ARG, "llama_moe_layer_workspace_size")
    return int(n)


def moe_layer_forward(cfg: LayerConfig, weights: dict, top_k: int, batch: Batch, hidden: torch.Tensor,
                      residual_in: Optional[torch.Tensor], residual_out: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, workspace: torch.Tensor, out_ids: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    """One Qwen3-MoE decoder layer; weights holds ln1, w_qkv, w_o, ln2 (as
    layer_forward) and w_router [E, H], w13 [E, 2I, H], w2 [E, H, I]; see
    llama_moe_layer_forward in the header."""
    c, b = cfg.c(), batch.c()
    E, H = weights["w_router"].shape
    m = LlamaMoeConfig(H, E, top_k, int(weights["w2"].shape[2]))
    w = LlamaMoeLayerWeights(_ptr(weights["ln1"]), _ptr(weights["w_qkv"]), _ptr(weights["w_o"]),
                             _ptr(weights["ln2"]), _ptr(weights["w_router"]), _ptr(weights["w13"]),
                             _ptr(weights["w2"]))
    st = lib().llama_moe_layer_forward(ctypes.byref(c), ctypes.byref(m), ctypes.byref(w), ctypes.byref(b),
                                       _ptr(hidden), _ptr(residual_in), _ptr(residual_out), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(out_ids), _ptr(workspace), workspace.numel(),
                                       _stream(stream))
    _check(st, "llama_moe_layer_forward")


def fold_norm_weights(norm_weight: torch.Tensor, w: torch.Tensor, out: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """bf16(w * norm_weight) column-wise, for a layer whose ln1/ln2 are None
    (the norm weights folded into w_qkv and w_gate_up)."""
    rows, cols = w.shape
    out = torch.empty_like(w) if out is None else out
    st = lib().llama_fold_norm_weights(_ptr(norm_weight), _ptr(w), rows, cols, _ptr(out), _stream(stream))
    _check(st, "llama_fold_norm_weights")
    return out


def folded_layer_weights(weights: dict, stream=None) -> dict:
    """The weights of a folded-norm layer: ln1/ln2 None, gamma folded into
    w_qkv and w_gate_up."""
    w = dict(weights)
    w["w_qkv"] = fold_norm_weights(weights["ln1"], weights["w_qkv"], stream=stream)
    w["w_gate_up"] = fold_norm_weights(weights["ln2"], weights["w_gate_up"], stream=stream)
    w["ln1"] = None
    w["ln2"] = None
    return w


def selftest_wait_timeout(stream=None) -> None:
    """Launches the bounded-wait self-test (a wait that runs out after ~2 s);
    llama_get_device_error then reports the timeout."""
    _check(lib().llama_selftest_wait_timeout(_stream(stream)), "llama_selftest_wait_timeout")


def launch_count() -> int:
    """Kernels launched through the library so far in this process."""
    return int(lib().llama_launch_count())
