// dsv4_static.cu -- dsv4_o_proj_static: the O-projection for callers that
// cannot allocate device memory (an engine plugin that owns no allocator, a
// latency path where cudaMalloc would synchronise the device).  The scratch
// that dsv4_o_proj takes from its caller lives here instead, in one file-scope
// device array of DSV4_STATIC_SCRATCH_BYTES that every device loading this
// library holds until the process exits.  Nothing here allocates.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/dsv4.h"
#include "dsv4_internal.h"

namespace {

// The scratch itself.  In host code its name is only a host-side stand-in for
// the symbol, not a device address: kernels get the address looked up below.
static __device__ __align__(256) uint8_t g_o_proj_scratch[DSV4_STATIC_SCRATCH_BYTES];

// The device address of the array, looked up once per device with that device
// current.  Only a successful lookup is kept; a failed one (say a first call
// made during stream capture) is tried again by the next call.
std::mutex g_setup_mutex;
std::atomic<bool> g_scratch_ready[dsv4::kMaxDevices];
void* g_scratch_addr[dsv4::kMaxDevices];

int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4_ERR_CUDA;
  if (dev < 0 || dev >= dsv4::kMaxDevices) return DSV4_ERR_UNSUPPORTED;
  if (!g_scratch_ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ready[dev].load(std::memory_order_relaxed)) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_o_proj_scratch) != cudaSuccess || p == nullptr)
        return DSV4_ERR_CUDA;
      g_scratch_addr[dev] = p;
      g_scratch_ready[dev].store(true, std::memory_order_release);
    }
  }
  *out = g_scratch_addr[dev];
  return DSV4_OK;
}

}  // namespace

extern "C" int dsv4_o_proj_static(const void* o, const int64_t* positions,
                                  const float* cos_sin_cache, int64_t max_pos,
                                  int64_t num_tokens, int n_groups, int heads_per_group,
                                  int nope_dim, int rope_dim, int quant_group_size,
                                  int o_lora_rank, int hidden, const void* wo_a_fp8,
                                  const uint8_t* wo_a_scale, const void* wo_b_fp8,
                                  const uint8_t* wo_b_scale, void* out, void* stream) {
  // Host validation of every argument first, with no CUDA call: without a
  // workspace the regular entry point reports the first argument error, or
  // DSV4_ERR_WORKSPACE when everything else is valid (DSV4_OK when T == 0).
  int rc = dsv4_o_proj_with_events(o, positions, cos_sin_cache, max_pos, num_tokens, n_groups,
                                   heads_per_group, nope_dim, rope_dim, quant_group_size,
                                   o_lora_rank, hidden, wo_a_fp8, wo_a_scale, wo_b_fp8,
                                   wo_b_scale, out, nullptr, 0, nullptr, stream);
  if (rc != DSV4_ERR_WORKSPACE) return rc;
  const size_t need = dsv4_o_proj_workspace_bytes(num_tokens, n_groups, heads_per_group,
                                                  nope_dim + rope_dim, o_lora_rank);
  if (need == 0 || need > DSV4_STATIC_SCRATCH_BYTES) return DSV4_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != DSV4_OK) return rc;
  return dsv4_o_proj_with_events(o, positions, cos_sin_cache, max_pos, num_tokens, n_groups,
                                 heads_per_group, nope_dim, rope_dim, quant_group_size,
                                 o_lora_rank, hidden, wo_a_fp8, wo_a_scale, wo_b_fp8, wo_b_scale,
                                 out, scratch, DSV4_STATIC_SCRATCH_BYTES, nullptr, stream);
}

extern "C" size_t dsv4_static_scratch_bytes(void) { return DSV4_STATIC_SCRATCH_BYTES; }
