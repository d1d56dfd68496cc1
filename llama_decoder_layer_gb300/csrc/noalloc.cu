// llama_paged_attention_noalloc: paged attention whose split-KV scratch lives
// in a fixed array inside this library instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory when they run
// attention.  Examples are a plugin whose host framework hands it only input
// and output buffers, and a process whose memory pool is owned and fenced by
// another runtime.  A third is a latency-critical loop that forbids
// allocation after start-up.  Such a caller has no way to provide the
// workspace that llama_paged_attention asks for.
//
// The array below is a file-scope device variable: every GPU that loads this
// library holds kNoAllocScratchBytes of it until the process exits.  Every
// call shares it, so calls that overlap on the GPU (different streams, or
// several host threads) race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "llama_layer.h"

// 32 MiB: the split-KV partials of B sequences whose contexts span C chunks
// of 1536 keys take B * C * n_heads * (head_dim + 2) * 4 bytes, plus a work
// list of 4 * (ceil(T/8) + B) bytes and 512 of alignment slack (256 for the
// partials' layout, 256 for aligning the scratch base): e.g. up to ~1000
// sequence-chunks at 64 heads x 128.
static constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;

static __device__ __align__(256) unsigned char llama_noalloc_attn_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch array for the current device.  In host code
// the array's name only stands in for the symbol; the address a kernel may use
// comes from cudaGetSymbolAddress, taken once per device with that device
// current.  Returns nullptr if the runtime call fails (its error is cleared, so
// the next launch does not pick it up).  The cached address belongs to the
// device's current context: after cudaDeviceReset the process must not call
// this entry point again on that device.
void* scratch_address() {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, llama_noalloc_attn_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" size_t llama_paged_attention_noalloc_limit(void) { return kNoAllocScratchBytes; }

extern "C" int llama_paged_attention_noalloc(const LlamaLayerConfig* cfg, const LlamaBatch* batch, const void* q,
                                             const void* k_cache, const void* v_cache, void* out,
                                             llama_stream_t stream) {
  // an invalid configuration or batch gets the status llama_paged_attention
  // would give it, before the size check
  const int st = llama::attention_args_status(cfg, batch);
  if (st != LLAMA_OK) return st;
  if (batch->num_tokens == 0) return LLAMA_OK;
  // the partials and work list (with their own 256-byte slack) plus 256 bytes
  // for aligning the base: what llama_paged_attention requires of a workspace
  const size_t need = llama::attn_partials_bytes(batch->num_seqs, batch->num_tokens, batch->max_seq_len,
                                                 cfg->n_heads, cfg->head_dim) +
                      256;
  if (need > kNoAllocScratchBytes) return LLAMA_ERR_SCRATCH_LIMIT;
  void* scratch = scratch_address();
  if (scratch == nullptr) return LLAMA_ERR_CUDA;
  // Nothing in the scratch has to start at zero: the combine step reads only
  // partials that the decode kernel wrote earlier in this same call, and the
  // prefill kernel reads only the work list the planning kernel wrote first.
  return llama_paged_attention(cfg, batch, q, k_cache, v_cache, out, scratch, kNoAllocScratchBytes, stream);
}
