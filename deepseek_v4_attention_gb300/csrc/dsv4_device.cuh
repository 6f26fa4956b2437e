// dsv4_device.cuh -- sm_103a device helpers for the O-projection kernels:
// mbarrier, TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, copy, load)
// written as inline PTX, plus the bounded waits every pipeline uses.
//
// Every wait on an mbarrier is bounded in time: after kWaitLimitNs it records
// DSV4_ERR_TIMEOUT in the device status word, raises the CTA's abort flag and
// returns false, so a broken pipeline ends the kernel instead of hanging it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsv4.h"

namespace dsv4 {

// Kernels receive the address of the library's device status word (a
// file-scope __device__ int, one per device) and record the first
// data-dependent error there; they never trap.
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if the
// CTA aborted (another role timed out) or this wait itself ran out of time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, int* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      record_status(status, DSV4_ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform wait: lane 0 owns the time limit, the other lanes wait for the
// phase or for the abort flag; the warp leaves together with one verdict, so
// a timeout can never split a warp in front of a shuffle or __syncwarp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, int* status) {
  bool done;
  if ((threadIdx.x & 31) == 0) {
    done = mbar_wait(bar, parity, abort_flag, status);
  } else {
    while (true) {
      if (mbar_try_wait(bar, parity)) { done = true; break; }
      if (*abort_flag) { done = false; break; }
    }
  }
  return __all_sync(0xFFFFFFFFu, done);
}

// Warp-uniform wait for roles that wait long and must not take issue slots
// from compute warps on the same scheduler: only lane 0 polls, sleeping
// `sleep_ns` between polls; the other lanes wait at the warp barrier.  Same
// time limit and abort rules as mbar_wait.
__device__ __forceinline__ bool mbar_wait_warp_lazy(uint64_t* bar, uint32_t parity,
                                                    volatile int* abort_flag, int* status,
                                                    unsigned sleep_ns) {
  int done = 1;
  if ((threadIdx.x & 31) == 0 && !mbar_try_wait(bar, parity)) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
      __nanosleep(sleep_ns);
      if (mbar_try_wait(bar, parity)) break;
      if (*abort_flag) { done = 0; break; }
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        record_status(status, DSV4_ERR_TIMEOUT);
        done = 0;
        break;
      }
    }
  }
  return __shfl_sync(0xFFFFFFFFu, done, 0) != 0;
}

// A shorter wait used only while draining after an abort.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 50000000ull) return false;  // 50 ms
  }
  return true;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Prefetch of a 2D box of a tensor into L2 (no shared memory, no completion
// to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// TMA store of a 2D box from this CTA's shared memory, tracked as a bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------- programmatic dependent launch --
// A kernel launched with programmatic stream serialization may start while the
// previous kernel of the stream still runs; griddep_wait() blocks until that
// kernel has completed and its memory is visible (a no-op for a normal launch).
// griddep_launch_dependents() lets the next such kernel start once every CTA of
// this grid has executed it (or exited).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- clusters --
__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// Cluster-wide barrier, executed per thread (every thread of every CTA of the
// cluster arrives once); release/acquire order shared::cluster accesses.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ------------------------------------------------- quantisation helpers --
// Shared by the quantiser and the GEMM's fused producer warps, so that both
// produce the same codes and scales bit for bit.

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Inverse rotation of one interleaved pair (a, b) by the angle with cosine c
// and sine s, in fp32 with a fixed order: each cross product is rounded first.
__device__ __forceinline__ void inv_rotate(float& a, float& b, float c, float s) {
  const float bs = __fmul_rn(b, s);
  const float as = __fmul_rn(a, s);
  const float y0 = __fmaf_rn(a, c, bs);
  const float y1 = __fmaf_rn(b, c, -as);
  a = y0;
  b = y1;
}

// Maximum over the 16 lanes of a half-warp.
__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

// ---------------------------------------------------------------- tcgen05 --
// Tensor-memory address: bits [31:16] lane, bits [15:0] column.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in
// bits [0,14), leading-dimension byte offset >> 4 in [16,30), stride-dimension
// byte offset >> 4 in [32,46), the fixed version field 1 in [46,48), base
// offset 0, swizzle mode in [61,64) (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
  return d;
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: E4M3 x E4M3,
// fp32 accumulate, both operands K-major, UE8M0 scale factors.
//   [4,6) scale-factor id of B, [7,10) A format (E4M3 = 0), [10,13) B format,
//   [15] A major, [16] B major, [17,23) N >> 3, [23] scale format (UE8M0 = 1),
//   [24,29) M >> 4, [29,31) scale-factor id of A.
__device__ __forceinline__ uint32_t mxf8_idesc(uint32_t M, uint32_t N, uint32_t sfa_id,
                                               uint32_t sfb_id) {
  uint32_t d = 0;
  d |= (sfb_id & 3u) << 4;
  d |= ((N >> 3) & 0x3Fu) << 17;
  d |= 1u << 23;
  d |= ((M >> 4) & 0x1Fu) << 24;
  d |= (sfa_id & 3u) << 29;
  return d;
}

__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulate,
// both K-major: [4,6) D format (F32 = 1), [7,10) A format (BF16 = 1),
// [10,13) B format (BF16 = 1), [17,23) N >> 3, [24,29) M >> 4.
__device__ __forceinline__ uint32_t bf16_idesc(uint32_t M, uint32_t N) {
  uint32_t d = 0;
  d |= 1u << 4;
  d |= 1u << 7;
  d |= 1u << 10;
  d |= ((N >> 3) & 0x3Fu) << 17;
  d |= ((M >> 4) & 0x1Fu) << 24;
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on an mbarrier once every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Shared memory -> tensor memory: 32 rows of 16 bytes, broadcast to the four
// 32-lane quarters of TMEM (4 consecutive 32-bit columns per lane).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------- number formats --
// UE8M0 exponent of a 128-element block: the smallest e with
// max(amax, 1e-4) <= 448 * 2^e.  With a = m * 2^E (m in [1, 2)) and
// 448 = 1.75 * 2^8 this is E - 8 when m <= 1.75 (mantissa field <= 0x600000),
// else E - 7.  Integer work on the fp32 bits only.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
  const float a = fmaxf(amax, 1e-4f);
  const uint32_t u = __float_as_uint(a);
  const int E = static_cast<int>(u >> 23) - 127;
  return ((u & 0x7FFFFFu) <= 0x600000u) ? E - 8 : E - 7;
}

// 2^-e as an fp32 (exact; e is within [-22, 121] here).
__device__ __forceinline__ float exp2_neg(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// Two fp32 -> two e4m3 (round to nearest even, saturate to +-448); the first
// argument lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Quantises 8 values with scale 2^e (inv_scale = 2^-e) into 8 e4m3 bytes.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float inv_scale) {
  uint2 r;
  r.x = static_cast<uint32_t>(e4m3x2(f[0] * inv_scale, f[1] * inv_scale)) |
        (static_cast<uint32_t>(e4m3x2(f[2] * inv_scale, f[3] * inv_scale)) << 16);
  r.y = static_cast<uint32_t>(e4m3x2(f[4] * inv_scale, f[5] * inv_scale)) |
        (static_cast<uint32_t>(e4m3x2(f[6] * inv_scale, f[7] * inv_scale)) << 16);
  return r;
}

}  // namespace dsv4
