// dsv4_api.cu -- the C ABI (include/dsv4.h): host-side validation, workspace
// carving and launches.  Nothing here allocates device memory or synchronises
// a stream, except dsv4_device_status(), whose job is to read the status word.
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/dsv4.h"
#include "dsv4_device.cuh"
#include "dsv4_internal.h"

namespace dsv4 {

// The device status word: one per device (a module-scope variable, so it exists
// on every device that loads this library without any run-time allocation).
__device__ int g_status_word = 0;

namespace {

// Diagnostics: one thread waits, with the pipelines' bounded wait, on an
// mbarrier that nothing ever arrives on.  The wait gives up after limit_ns,
// records DSV4_ERR_TIMEOUT and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    (void)mbar_wait(&bar, 0, &abort_flag, status, limit_ns);  // phase 0 never completes
  }
  __syncthreads();
}

// Per-device facts, looked up on the first call with that device current.
// Only a complete lookup is kept: a failure is returned and tried again by the
// next call.
std::mutex g_device_mutex;
std::atomic<bool> g_device_ready[kMaxDevices];
DeviceInfo g_devices[kMaxDevices];

thread_local int t_last_launches = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

int64_t tma_aligned_tokens(int64_t T) { return (T + 3) / 4 * 4; }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

int check_quant_shapes(int64_t T, int64_t max_pos, int n_groups, int hpg, int nope, int rope,
                       int qgs) {
  if (T < 0 || n_groups <= 0 || hpg <= 0 || qgs <= 0 || nope < 0 || rope < 0)
    return DSV4_ERR_SHAPE;
  const int head_dim = nope + rope;
  // the asserts of fused_inv_rope_fp8_quant (H == G * hpg holds by construction here)
  if (head_dim % qgs != 0) return DSV4_ERR_SHAPE;
  if (nope % qgs != qgs - rope) return DSV4_ERR_SHAPE;
  if (rope % 2 != 0) return DSV4_ERR_SHAPE;
  if (max_pos <= 0) return DSV4_ERR_SHAPE;
  if (static_cast<int64_t>(n_groups) * hpg > (1 << 20)) return DSV4_ERR_SHAPE;
  return DSV4_OK;
}

int check_quant_supported(int nope, int rope, int qgs) {
  if (nope != 448 || rope != 64 || qgs != 128) return DSV4_ERR_UNSUPPORTED;
  return DSV4_OK;
}

}  // namespace

int get_device_info(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSV4_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSV4_ERR_UNSUPPORTED;
  if (!g_device_ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_device_mutex);
    if (!g_device_ready[dev].load(std::memory_order_relaxed)) {
      DeviceInfo d;
      d.device = dev;
      int v = 0;
      if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
              cudaSuccess ||
          cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
              cudaSuccess ||
          cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
              cudaSuccess ||
          cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
              cudaSuccess)
        return DSV4_ERR_CUDA;
      d.max_smem_optin = static_cast<size_t>(v);
      // the library carries sm_103a code only
      if (d.cc_major != 10 || d.cc_minor != 3) return DSV4_ERR_UNSUPPORTED;
      void* sym = nullptr;
      if (cudaGetSymbolAddress(&sym, g_status_word) != cudaSuccess || sym == nullptr)
        return DSV4_ERR_CUDA;
      d.status = static_cast<int*>(sym);
      g_devices[dev] = d;
      g_device_ready[dev].store(true, std::memory_order_release);
    }
  }
  *out = g_devices[dev];
  return DSV4_OK;
}

}  // namespace dsv4

using namespace dsv4;

extern "C" {

const char* dsv4_status_string(int status) {
  switch (status) {
    case DSV4_OK: return "DSV4_OK";
    case DSV4_ERR_SHAPE: return "DSV4_ERR_SHAPE: invalid sizes";
    case DSV4_ERR_NULL: return "DSV4_ERR_NULL: null pointer";
    case DSV4_ERR_ALIGN: return "DSV4_ERR_ALIGN: misaligned pointer";
    case DSV4_ERR_UNSUPPORTED: return "DSV4_ERR_UNSUPPORTED: device or parameter not supported";
    case DSV4_ERR_WORKSPACE: return "DSV4_ERR_WORKSPACE: workspace missing or too small";
    case DSV4_ERR_CUDA: return "DSV4_ERR_CUDA: CUDA call failed";
    case DSV4_ERR_TIMEOUT: return "DSV4_ERR_TIMEOUT: a kernel pipeline wait timed out";
    case DSV4_ERR_RANGE: return "DSV4_ERR_RANGE: position outside [0, max_pos)";
    default: return "unknown dsv4 status";
  }
}

int dsv4_last_launch_count(void) { return t_last_launches; }

int dsv4_inv_rope_fp8_quant(const void* o, const int64_t* positions, const float* cos_sin_cache,
                            int64_t num_tokens, int64_t max_pos, int n_groups,
                            int heads_per_group, int nope_dim, int rope_dim,
                            int quant_group_size, void* out_fp8, int32_t* out_scale,
                            void* stream) {
  t_last_launches = 0;
  int rc = check_quant_shapes(num_tokens, max_pos, n_groups, heads_per_group, nope_dim, rope_dim,
                              quant_group_size);
  if (rc != DSV4_OK) return rc;
  if ((rc = check_quant_supported(nope_dim, rope_dim, quant_group_size)) != DSV4_OK) return rc;
  if (num_tokens == 0) return DSV4_OK;
  if (!o || !positions || !cos_sin_cache || !out_fp8 || !out_scale) return DSV4_ERR_NULL;
  if (!aligned16(o) || !aligned16(positions) || !aligned16(cos_sin_cache) ||
      !aligned16(out_fp8) || !aligned16(out_scale))
    return DSV4_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = get_device_info(&dev)) != DSV4_OK) return rc;
  rc = launch_inv_rope_fp8_quant(o, positions, cos_sin_cache, num_tokens, max_pos, n_groups,
                                 heads_per_group, out_fp8, out_scale,
                                 static_cast<cudaStream_t>(stream), dev);
  if (rc == DSV4_OK) t_last_launches = 1;
  return rc;
}

int dsv4_grouped_wo_a(const void* x_fp8, const int32_t* x_scale, int64_t num_tokens,
                      int n_groups, int group_dim, int o_lora_rank, const void* w_fp8,
                      const uint8_t* w_scale, void* z, void* stream) {
  return dsv4_grouped_wo_a_ex(x_fp8, x_scale, num_tokens, n_groups, group_dim, o_lora_rank, w_fp8,
                              w_scale, z, 0u, stream);
}

int dsv4_grouped_wo_a_ex(const void* x_fp8, const int32_t* x_scale, int64_t num_tokens,
                         int n_groups, int group_dim, int o_lora_rank, const void* w_fp8,
                         const uint8_t* w_scale, void* z, unsigned flags, void* stream) {
  t_last_launches = 0;
  if ((flags & ~DSV4_OVERLAP_PREVIOUS) != 0) return DSV4_ERR_SHAPE;
  if (num_tokens < 0 || n_groups <= 0 || group_dim <= 0 || o_lora_rank <= 0 ||
      group_dim % 128 != 0 || o_lora_rank % 128 != 0)
    return DSV4_ERR_SHAPE;
  if (num_tokens == 0) return DSV4_OK;
  if (!x_fp8 || !x_scale || !w_fp8 || !w_scale || !z) return DSV4_ERR_NULL;
  if (!aligned16(x_fp8) || !aligned16(x_scale) || !aligned16(w_fp8) || !aligned16(z))
    return DSV4_ERR_ALIGN;
  if (num_tokens > (int64_t(1) << 31) - 128) return DSV4_ERR_SHAPE;
  DeviceInfo dev;
  int rc = get_device_info(&dev);
  if (rc != DSV4_OK) return rc;
  GemmProblem p;
  p.T = num_tokens;
  p.G = n_groups;
  p.N = o_lora_rank;
  p.K = group_dim;
  p.a = x_fp8;
  p.a_scale = x_scale;
  p.b = w_fp8;
  p.b_scale = w_scale;
  p.epilogue = kEpiBf16;
  p.out_bf16 = z;
  p.after_own_kernel = (flags & DSV4_OVERLAP_PREVIOUS) != 0;
  rc = launch_block_scaled_gemm(p, static_cast<cudaStream_t>(stream), dev);
  if (rc == DSV4_OK) t_last_launches = 1;
  return rc;
}

int dsv4_inv_rope_grouped_wo_a(const void* o, const int64_t* positions,
                               const float* cos_sin_cache, int64_t num_tokens, int64_t max_pos,
                               int n_groups, int heads_per_group, int nope_dim, int rope_dim,
                               int quant_group_size, int o_lora_rank, const void* w_fp8,
                               const uint8_t* w_scale, void* z, void* stream) {
  t_last_launches = 0;
  int rc = check_quant_shapes(num_tokens, max_pos, n_groups, heads_per_group, nope_dim, rope_dim,
                              quant_group_size);
  if (rc != DSV4_OK) return rc;
  if (o_lora_rank <= 0 || o_lora_rank % 128 != 0) return DSV4_ERR_SHAPE;
  if ((rc = check_quant_supported(nope_dim, rope_dim, quant_group_size)) != DSV4_OK) return rc;
  if (num_tokens == 0) return DSV4_OK;
  if (num_tokens > DSV4_FUSED_MAX_TOKENS || max_pos > INT32_MAX) return DSV4_ERR_UNSUPPORTED;
  if (!o || !positions || !cos_sin_cache || !w_fp8 || !w_scale || !z) return DSV4_ERR_NULL;
  if (!aligned16(o) || !aligned16(positions) || !aligned16(cos_sin_cache) || !aligned16(w_fp8) ||
      !aligned16(z))
    return DSV4_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = get_device_info(&dev)) != DSV4_OK) return rc;
  GemmProblem p;
  p.T = num_tokens;
  p.G = n_groups;
  p.N = o_lora_rank;
  p.K = heads_per_group * (nope_dim + rope_dim);
  p.b = w_fp8;
  p.b_scale = w_scale;
  p.epilogue = kEpiBf16;
  p.out_bf16 = z;
  p.fused_a = true;
  p.o = static_cast<const uint16_t*>(o);
  p.positions = positions;
  p.cache = cos_sin_cache;
  p.max_pos = max_pos;
  p.heads = n_groups * heads_per_group;
  p.heads_per_group = heads_per_group;
  rc = launch_block_scaled_gemm(p, static_cast<cudaStream_t>(stream), dev);
  if (rc == DSV4_OK) t_last_launches = 1;
  return rc;
}

int dsv4_inv_rope_bf16(const void* o, const int64_t* positions, const float* cos_sin_cache,
                       int64_t num_tokens, int64_t max_pos, int n_groups, int heads_per_group,
                       int nope_dim, int rope_dim, void* out_bf16, void* stream) {
  t_last_launches = 0;
  int rc = check_quant_shapes(num_tokens, max_pos, n_groups, heads_per_group, nope_dim, rope_dim,
                              128);
  if (rc != DSV4_OK) return rc;
  if ((rc = check_quant_supported(nope_dim, rope_dim, 128)) != DSV4_OK) return rc;
  if (num_tokens == 0) return DSV4_OK;
  if (!o || !positions || !cos_sin_cache || !out_bf16) return DSV4_ERR_NULL;
  if (!aligned16(o) || !aligned16(positions) || !aligned16(cos_sin_cache) || !aligned16(out_bf16))
    return DSV4_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = get_device_info(&dev)) != DSV4_OK) return rc;
  rc = launch_inv_rope_bf16(o, positions, cos_sin_cache, num_tokens, max_pos, n_groups,
                            heads_per_group, out_bf16, static_cast<cudaStream_t>(stream), dev);
  if (rc == DSV4_OK) t_last_launches = 1;
  return rc;
}

int dsv4_grouped_wo_a_bf16(const void* x_bf16, int64_t num_tokens, int n_groups, int group_dim,
                           int o_lora_rank, const void* w_bf16, void* z, void* stream) {
  t_last_launches = 0;
  if (num_tokens < 0 || n_groups <= 0 || group_dim <= 0 || o_lora_rank <= 0 ||
      group_dim % 64 != 0 || o_lora_rank % 128 != 0)
    return DSV4_ERR_SHAPE;
  if (num_tokens == 0) return DSV4_OK;
  if (!x_bf16 || !w_bf16 || !z) return DSV4_ERR_NULL;
  if (!aligned16(x_bf16) || !aligned16(w_bf16) || !aligned16(z)) return DSV4_ERR_ALIGN;
  if (num_tokens > (int64_t(1) << 31) - 128) return DSV4_ERR_SHAPE;
  DeviceInfo dev;
  int rc = get_device_info(&dev);
  if (rc != DSV4_OK) return rc;
  GemmProblem p;
  p.T = num_tokens;
  p.G = n_groups;
  p.N = o_lora_rank;
  p.K = group_dim;
  p.a = x_bf16;
  p.b = w_bf16;
  p.bf16 = true;
  p.epilogue = kEpiBf16;
  p.out_bf16 = z;
  rc = launch_block_scaled_gemm(p, static_cast<cudaStream_t>(stream), dev);
  if (rc == DSV4_OK) t_last_launches = 1;
  return rc;
}

size_t dsv4_o_proj_workspace_bytes(int64_t num_tokens, int n_groups, int heads_per_group,
                                   int head_dim, int o_lora_rank) {
  if (num_tokens < 0 || n_groups <= 0 || heads_per_group <= 0 || head_dim <= 0 ||
      head_dim % 128 != 0 || o_lora_rank <= 0 || o_lora_rank % 128 != 0)
    return 0;
  const int64_t T = num_tokens;
  const int64_t T_al = tma_aligned_tokens(T);
  const int64_t D = static_cast<int64_t>(heads_per_group) * head_dim;
  const int64_t PK = (D / 128 + 3) / 4;
  const int64_t C = static_cast<int64_t>(n_groups) * o_lora_rank;
  const int64_t PKC = (C / 128 + 3) / 4;
  size_t bytes = 0;
  bytes += round256(static_cast<size_t>(n_groups) * T * D);        // x codes
  bytes += round256(static_cast<size_t>(n_groups) * PK * T_al * 4); // x scales
  bytes += round256(static_cast<size_t>(T) * C);                    // zq codes
  bytes += round256(static_cast<size_t>(PKC) * T_al * 4);           // zq scales
  return bytes == 0 ? 256 : bytes;
}

}  // extern "C"

namespace {

// The quantiser's outputs and the re-quantised z inside a dsv4_o_proj
// workspace: four parts, each starting at a 256-byte boundary (include/dsv4.h).
struct OProjWorkspace {
  uint8_t* x;
  int32_t* xs;
  uint8_t* zq;
  int32_t* zs;
};

OProjWorkspace carve_workspace(void* workspace, int64_t T, int n_groups, int64_t D,
                               int o_lora_rank) {
  const int64_t T_al = tma_aligned_tokens(T);
  const int64_t PK = (D / 128 + 3) / 4;
  const int64_t C = static_cast<int64_t>(n_groups) * o_lora_rank;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  OProjWorkspace w;
  w.x = ws;
  ws += round256(static_cast<size_t>(n_groups) * T * D);
  w.xs = reinterpret_cast<int32_t*>(ws);
  ws += round256(static_cast<size_t>(n_groups) * PK * T_al * 4);
  w.zq = ws;
  ws += round256(static_cast<size_t>(T) * C);
  w.zs = reinterpret_cast<int32_t*>(ws);
  return w;
}

// wo_a with the fused z re-quantisation into zq / zs, then wo_b into `out`
// (bf16, or the fp32 partial sums of a group range).  `overlap`: the GEMMs may
// start under the previous kernel of the stream (programmatic launch).
int o_proj_gemms(const void* x, const int32_t* xs, int64_t T, int n_groups, int64_t D,
                 int o_lora_rank, int hidden, const void* wo_a_fp8, const uint8_t* wo_a_scale,
                 const void* wo_b_fp8, const uint8_t* wo_b_scale, void* out, bool out_f32,
                 uint8_t* zq, int32_t* zs, bool overlap, void* const* stage_events,
                 cudaStream_t s, const DeviceInfo& dev) {
  auto mark = [&](int i) {
    if (!stage_events) return true;
    return cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s) == cudaSuccess;
  };
  GemmProblem a;
  a.T = T;
  a.G = n_groups;
  a.N = o_lora_rank;
  a.K = static_cast<int>(D);
  a.a = x;
  a.a_scale = xs;
  a.b = wo_a_fp8;
  a.b_scale = wo_a_scale;
  a.epilogue = kEpiQuant;
  a.q_out = zq;
  a.q_scale = zs;
  a.after_own_kernel = overlap;
  int rc = launch_block_scaled_gemm(a, s, dev);
  if (rc != DSV4_OK) return rc;
  if (!mark(2)) return DSV4_ERR_CUDA;

  GemmProblem b;
  b.T = T;
  b.G = 1;
  b.N = hidden;
  b.K = n_groups * o_lora_rank;
  b.a = zq;
  b.a_scale = zs;
  b.b = wo_b_fp8;
  b.b_scale = wo_b_scale;
  if (out_f32) {
    b.epilogue = kEpiF32;
    b.out_f32 = static_cast<float*>(out);
  } else {
    b.epilogue = kEpiBf16;
    b.out_bf16 = out;
  }
  b.after_own_kernel = overlap;
  if ((rc = launch_block_scaled_gemm(b, s, dev)) != DSV4_OK) return rc;
  if (!mark(3)) return DSV4_ERR_CUDA;
  return DSV4_OK;
}

// dsv4_o_proj, dsv4_o_proj_with_events and dsv4_o_proj_partial.
int o_proj(const void* o, const int64_t* positions, const float* cos_sin_cache, int64_t max_pos,
           int64_t num_tokens, int n_groups, int heads_per_group, int nope_dim, int rope_dim,
           int quant_group_size, int o_lora_rank, int hidden, const void* wo_a_fp8,
           const uint8_t* wo_a_scale, const void* wo_b_fp8, const uint8_t* wo_b_scale,
           void* out, bool out_f32, void* workspace, size_t workspace_bytes,
           void* const* stage_events, void* stream) {
  t_last_launches = 0;
  int rc = check_quant_shapes(num_tokens, max_pos, n_groups, heads_per_group, nope_dim, rope_dim,
                              quant_group_size);
  if (rc != DSV4_OK) return rc;
  if (o_lora_rank <= 0 || o_lora_rank % 128 != 0 || hidden <= 0 || hidden % 128 != 0)
    return DSV4_ERR_SHAPE;
  if ((rc = check_quant_supported(nope_dim, rope_dim, quant_group_size)) != DSV4_OK) return rc;
  if (num_tokens == 0) return DSV4_OK;
  if (num_tokens > (int64_t(1) << 31) - 128) return DSV4_ERR_SHAPE;
  if (!o || !positions || !cos_sin_cache || !wo_a_fp8 || !wo_a_scale || !wo_b_fp8 ||
      !wo_b_scale || !out)
    return DSV4_ERR_NULL;
  if (!aligned16(o) || !aligned16(positions) || !aligned16(cos_sin_cache) ||
      !aligned16(wo_a_fp8) || !aligned16(wo_b_fp8) || !aligned16(out))
    return DSV4_ERR_ALIGN;
  const int head_dim = nope_dim + rope_dim;
  const size_t need =
      dsv4_o_proj_workspace_bytes(num_tokens, n_groups, heads_per_group, head_dim, o_lora_rank);
  if (!workspace || workspace_bytes < need) return DSV4_ERR_WORKSPACE;
  if (!aligned256(workspace)) return DSV4_ERR_ALIGN;

  DeviceInfo dev;
  if ((rc = get_device_info(&dev)) != DSV4_OK) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t D = static_cast<int64_t>(heads_per_group) * head_dim;
  const OProjWorkspace w = carve_workspace(workspace, num_tokens, n_groups, D, o_lora_rank);

  if (stage_events &&
      cudaEventRecord(static_cast<cudaEvent_t>(stage_events[0]), s) != cudaSuccess)
    return DSV4_ERR_CUDA;
  rc = launch_inv_rope_fp8_quant(o, positions, cos_sin_cache, num_tokens, max_pos, n_groups,
                                 heads_per_group, w.x, w.xs, s, dev);
  if (rc != DSV4_OK) return rc;
  if (stage_events &&
      cudaEventRecord(static_cast<cudaEvent_t>(stage_events[1]), s) != cudaSuccess)
    return DSV4_ERR_CUDA;
  // Programmatic launches overlap a GEMM's prologue (and, on one SM, its first
  // weight loads) with the previous kernel's tail: measured -2 % time at
  // T <= 512, -1.0 % at T = 4096 and -1.4 % at T = 8192; never when stage
  // events are asked for, whose per-kernel times would then overlap.
  const bool overlap = stage_events == nullptr;
  rc = o_proj_gemms(w.x, w.xs, num_tokens, n_groups, D, o_lora_rank, hidden, wo_a_fp8,
                    wo_a_scale, wo_b_fp8, wo_b_scale, out, out_f32, w.zq, w.zs, overlap,
                    stage_events, s, dev);
  if (rc != DSV4_OK) return rc;
  t_last_launches = 3;
  return DSV4_OK;
}

}  // namespace

extern "C" {

int dsv4_o_proj(const void* o, const int64_t* positions, const float* cos_sin_cache,
                int64_t max_pos, int64_t num_tokens, int n_groups, int heads_per_group,
                int nope_dim, int rope_dim, int quant_group_size, int o_lora_rank, int hidden,
                const void* wo_a_fp8, const uint8_t* wo_a_scale, const void* wo_b_fp8,
                const uint8_t* wo_b_scale, void* out, void* workspace, size_t workspace_bytes,
                void* stream) {
  return o_proj(o, positions, cos_sin_cache, max_pos, num_tokens, n_groups, heads_per_group,
                nope_dim, rope_dim, quant_group_size, o_lora_rank, hidden, wo_a_fp8, wo_a_scale,
                wo_b_fp8, wo_b_scale, out, false, workspace, workspace_bytes, nullptr, stream);
}

int dsv4_o_proj_with_events(const void* o, const int64_t* positions, const float* cos_sin_cache,
                            int64_t max_pos, int64_t num_tokens, int n_groups,
                            int heads_per_group, int nope_dim, int rope_dim,
                            int quant_group_size, int o_lora_rank, int hidden,
                            const void* wo_a_fp8, const uint8_t* wo_a_scale,
                            const void* wo_b_fp8, const uint8_t* wo_b_scale, void* out,
                            void* workspace, size_t workspace_bytes, void* const* stage_events,
                            void* stream) {
  return o_proj(o, positions, cos_sin_cache, max_pos, num_tokens, n_groups, heads_per_group,
                nope_dim, rope_dim, quant_group_size, o_lora_rank, hidden, wo_a_fp8, wo_a_scale,
                wo_b_fp8, wo_b_scale, out, false, workspace, workspace_bytes, stage_events,
                stream);
}

int dsv4_o_proj_partial(const void* o, const int64_t* positions, const float* cos_sin_cache,
                        int64_t max_pos, int64_t num_tokens, int n_groups, int heads_per_group,
                        int nope_dim, int rope_dim, int quant_group_size, int o_lora_rank,
                        int hidden, const void* wo_a_fp8, const uint8_t* wo_a_scale,
                        const void* wo_b_fp8, const uint8_t* wo_b_scale, float* out_partial,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return o_proj(o, positions, cos_sin_cache, max_pos, num_tokens, n_groups, heads_per_group,
                nope_dim, rope_dim, quant_group_size, o_lora_rank, hidden, wo_a_fp8, wo_a_scale,
                wo_b_fp8, wo_b_scale, out_partial, true, workspace, workspace_bytes, nullptr,
                stream);
}

int dsv4_sum_partials(const float* const* partials, int n_partials, int64_t num_elems,
                      void* out_bf16, void* stream) {
  t_last_launches = 0;
  if (n_partials < 1 || n_partials > DSV4_MAX_PARTIALS || num_elems < 0) return DSV4_ERR_SHAPE;
  if (num_elems == 0) return DSV4_OK;
  if (!partials || !out_bf16) return DSV4_ERR_NULL;
  for (int j = 0; j < n_partials; ++j) {
    if (!partials[j]) return DSV4_ERR_NULL;
    if (!aligned16(partials[j])) return DSV4_ERR_ALIGN;
  }
  if (!aligned16(out_bf16)) return DSV4_ERR_ALIGN;
  DeviceInfo dev;
  int rc = get_device_info(&dev);
  if (rc != DSV4_OK) return rc;
  rc = launch_sum_partials(partials, n_partials, num_elems, out_bf16,
                           static_cast<cudaStream_t>(stream), dev);
  if (rc == DSV4_OK) t_last_launches = 1;
  return rc;
}

int dsv4_rope_quant_unsupported_reason(int n_local_heads, int kv_cache_fp8, int wo_a_fp8,
                                       const char** reason) {
  const char* why = nullptr;
  if (n_local_heads != DSV4_ROPE_QUANT_NUM_HEADS)
    why = "the fused inverse-RoPE + FP8 attention output is laid out for exactly 128 local "
          "query heads; padding a smaller head count up to it costs more attention work "
          "than the fusion saves";
  else if (!kv_cache_fp8)
    why = "the fused attention output is produced only with the per-tensor FP8 KV cache";
  else if (!wo_a_fp8)
    why = "a pre-quantised attention output needs an FP8 wo_a";
  if (reason) *reason = why;
  return why ? DSV4_ERR_UNSUPPORTED : DSV4_OK;
}

size_t dsv4_o_proj_prequant_workspace_bytes(int64_t num_tokens, int n_groups, int o_lora_rank) {
  if (num_tokens < 0 || n_groups <= 0 || o_lora_rank <= 0 || o_lora_rank % 128 != 0) return 0;
  const int64_t C = static_cast<int64_t>(n_groups) * o_lora_rank;
  const int64_t PKC = (C / 128 + 3) / 4;
  const size_t bytes = round256(static_cast<size_t>(num_tokens) * C) +
                       round256(static_cast<size_t>(PKC) * tma_aligned_tokens(num_tokens) * 4);
  return bytes == 0 ? 256 : bytes;
}

int dsv4_o_proj_prequant(const void* x_fp8, const int32_t* x_scale, int64_t num_tokens,
                         int n_slots, int n_groups, int group_dim, int o_lora_rank, int hidden,
                         const void* wo_a_fp8, const uint8_t* wo_a_scale, const void* wo_b_fp8,
                         const uint8_t* wo_b_scale, void* out, void* workspace,
                         size_t workspace_bytes, void* stream) {
  t_last_launches = 0;
  if (num_tokens < 0 || n_groups <= 0 || n_slots < n_groups || group_dim <= 0 ||
      group_dim % 128 != 0 || o_lora_rank <= 0 || o_lora_rank % 128 != 0 || hidden <= 0 ||
      hidden % 128 != 0)
    return DSV4_ERR_SHAPE;
  if (num_tokens == 0) return DSV4_OK;
  if (num_tokens > (int64_t(1) << 31) - 128) return DSV4_ERR_SHAPE;
  if (!x_fp8 || !x_scale || !wo_a_fp8 || !wo_a_scale || !wo_b_fp8 || !wo_b_scale || !out)
    return DSV4_ERR_NULL;
  if (!aligned16(x_fp8) || !aligned16(x_scale) || !aligned16(wo_a_fp8) || !aligned16(wo_b_fp8) ||
      !aligned16(out))
    return DSV4_ERR_ALIGN;
  const size_t need = dsv4_o_proj_prequant_workspace_bytes(num_tokens, n_groups, o_lora_rank);
  if (!workspace || workspace_bytes < need) return DSV4_ERR_WORKSPACE;
  if (!aligned256(workspace)) return DSV4_ERR_ALIGN;
  DeviceInfo dev;
  int rc = get_device_info(&dev);
  if (rc != DSV4_OK) return rc;
  // The live groups are the first n_groups slots: a prefix of the group-major
  // codes [slot][T][D] and of the scales [slot][PK][T_al].
  uint8_t* zq = static_cast<uint8_t*>(workspace);
  int32_t* zs = reinterpret_cast<int32_t*>(
      zq + round256(static_cast<size_t>(num_tokens) * n_groups * o_lora_rank));
  rc = o_proj_gemms(x_fp8, x_scale, num_tokens, n_groups, group_dim, o_lora_rank, hidden,
                    wo_a_fp8, wo_a_scale, wo_b_fp8, wo_b_scale, out, false, zq, zs,
                    false, nullptr, static_cast<cudaStream_t>(stream), dev);
  if (rc != DSV4_OK) return rc;
  t_last_launches = 2;
  return DSV4_OK;
}

int dsv4_selftest_wait_timeout(int64_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return DSV4_ERR_SHAPE;
  DeviceInfo dev;
  int rc = get_device_info(&dev);
  if (rc != DSV4_OK) return rc;
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_us) * 1000u, dev.status);
  return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

int dsv4_device_status(void* stream, int clear) {
  DeviceInfo dev;
  int rc = get_device_info(&dev);
  if (rc != DSV4_OK) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSV4_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSV4_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpy(dev.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return DSV4_ERR_CUDA;
  }
  return v;
}

}  // extern "C"
