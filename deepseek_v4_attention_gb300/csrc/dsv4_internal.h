// dsv4_internal.h -- declarations shared by the library's translation units
// (host side only; no device code here).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace dsv4 {

constexpr int kMaxDevices = 64;

// Host state computed once per device on first use (a function attribute set,
// an occupancy figure): thread-safe, and only a success is kept, so a failed
// first attempt (a transient error, a call made during stream capture) is
// retried by the next call instead of being remembered.  `compute` returns a
// positive value on success.
inline std::mutex& lazy_state_mutex() {
  static std::mutex m;
  return m;
}

template <class F>
int lazy_per_device(std::atomic<int> (&slots)[kMaxDevices], int device, F compute) {
  if (device < 0 || device >= kMaxDevices) return 0;
  int v = slots[device].load(std::memory_order_acquire);
  if (v > 0) return v;
  std::lock_guard<std::mutex> lock(lazy_state_mutex());
  v = slots[device].load(std::memory_order_relaxed);
  if (v > 0) return v;
  v = compute();
  if (v > 0) slots[device].store(v, std::memory_order_release);
  return v;
}

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int cc_major = 0;
  int cc_minor = 0;
  size_t max_smem_optin = 0;
  int* status = nullptr;  // device address of the status word on this device
};

// Epilogue of the block-scaled GEMM.
enum GemmEpilogue : int {
  kEpiBf16 = 0,   // store fp32 accumulators as bf16 rows [T][G*N]
  kEpiQuant = 1,  // round to bf16, then per-128 UE8M0 FP8 re-quantisation of each row
  kEpiF32 = 2,    // store the fp32 accumulators as they are, rows [T][G*N]
};

struct GemmProblem {
  int64_t T = 0;          // rows (tokens)
  int G = 1;              // groups: group g of A meets rows g*N:(g+1)*N of B
  int N = 0;              // output columns per group (multiple of 128)
  int K = 0;              // reduction length (multiple of 128)
  const void* a = nullptr;          // e4m3 (or bf16) physical [G][T][K]
  const int32_t* a_scale = nullptr; // int32 physical [G][ceil(K/512)][T_al]
  const void* b = nullptr;          // e4m3 [G*N][K] row-major
  const uint8_t* b_scale = nullptr; // UE8M0 bytes [G*N/128][K/128]
  int epilogue = kEpiBf16;
  bool bf16 = false;                // A and B bf16, no scales (kind::f16), K % 64 == 0
  bool after_own_kernel = false;    // the previous kernel on the stream does not write the
                                    // weights (b, b_scale): launch with programmatic stream
                                    // serialization and read them before it completes
  // Fused A (decode sizes, T <= 64): the kernel's producer warps build A from
  // the attention output (inverse rotation + per-128 FP8 quantisation, the
  // quantiser's arithmetic) instead of reading a pre-quantised a / a_scale;
  // K = heads_per_group * 512.
  bool fused_a = false;
  const uint16_t* o = nullptr;      // bf16 [T][heads][512]
  const int64_t* positions = nullptr;
  const float* cache = nullptr;     // fp32 [max_pos][64], cos || sin
  int64_t max_pos = 0;
  int heads = 0;                    // G * heads_per_group
  int heads_per_group = 0;
  void* out_bf16 = nullptr;         // bf16 [T][G*N] (kEpiBf16)
  float* out_f32 = nullptr;         // fp32 [T][G*N] (kEpiF32)
  uint8_t* q_out = nullptr;         // e4m3 [T][G*N]           (kEpiQuant)
  int32_t* q_scale = nullptr;       // int32 [ceil(G*N/512)][T_al] (kEpiQuant)
};

int get_device_info(DeviceInfo* out);

int launch_inv_rope_fp8_quant(const void* o, const int64_t* positions, const float* cache,
                              int64_t T, int64_t max_pos, int n_groups, int hpg, void* out_fp8,
                              int32_t* out_scale, cudaStream_t stream, const DeviceInfo& dev);

int launch_inv_rope_bf16(const void* o, const int64_t* positions, const float* cache, int64_t T,
                         int64_t max_pos, int n_groups, int hpg, void* out, cudaStream_t stream,
                         const DeviceInfo& dev);

int launch_block_scaled_gemm(const GemmProblem& p, cudaStream_t stream, const DeviceInfo& dev);

// The CTA-pair GEMM (dsv4_gemm_pair.cu): 256 x 256 tiles on two SMs, for the
// large shapes; eligible: A from memory (FP8, or bf16 with the bf16
// epilogue), N % 256 == 0, more than 128 tokens and at least one pair tile
// per two SMs.
bool pair_gemm_eligible(const GemmProblem& p, const DeviceInfo& dev);
int launch_pair_gemm(const GemmProblem& p, cudaStream_t stream, const DeviceInfo& dev);

// out[i] = bf16(sum over j < n of parts[j][i]), summed in fp32 in the order j = 0, 1, ...
int launch_sum_partials(const float* const* parts, int n, int64_t elems, void* out_bf16,
                        cudaStream_t stream, const DeviceInfo& dev);

}  // namespace dsv4
