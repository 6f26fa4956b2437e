// dsv4_quant.cu -- fused inverse RoPE + block-scaled FP8 quantisation
// (vLLM docs, models/deepseek_v4/common/ops/fused_inv_rope_fp8_quant, with the
// SM100-family packed UE8M0 scale layout).
//
// Work unit: one (token t, head h) pair = 512 bf16 = 1 KiB in, 512 B of e4m3
// + one packed int32 out.  One warp per unit; lane l holds elements
// [8l, 8l+8) and [256+8l, 256+8l+8) as two 16-byte loads, so each load
// instruction of the warp reads 512 contiguous bytes.
//   - 128-element blocks: lanes 0-15 / 16-31 of the first vector are blocks
//     0 / 1 of the head, of the second vector blocks 2 / 3; a block's amax is
//     a 4-step xor-shuffle inside one half-warp.
//   - the 64 rope lanes (head offsets 448..511) are lanes 24-31 of the second
//     vector; an interleaved pair (2i, 2i+1) never straddles a 16-byte vector,
//     so the rotation needs no shuffle.  Those lanes read cos[4(l-24)..+3] and
//     sin[4(l-24)..+3] of row positions[t] as two float4 loads.
//   - rotation in fp32 with a fixed order: y0 = fma(a, c, b*s),
//     y1 = fma(b, c, -(a*s)), each cross product rounded first.
//   - exponent from the fp32 bits of the amax (no log, no division);
//     q = y * 2^-e is exact; cvt.rn.satfinite to e4m3.
// Work is walked by a grid-stride loop in (t, h) order, so consecutive warps
// stream consecutive KiB of o; a warp takes kU heads of one token at a time,
// loads all of them before using any, and reads the position and the cos/sin
// row once for the kU heads.
#include "dsv4_device.cuh"
#include "dsv4_internal.h"

namespace dsv4 {

namespace {

constexpr int kHeadDim = 512;
constexpr int kRope = 64;

// One warp iteration = kU consecutive heads of one token (H % kU == 0): the
// position and the cos/sin row are loaded once for the kU heads, and all 2*kU
// 16-byte loads of o are issued before any value is used.
template <int kU>
__global__ void __launch_bounds__(256) inv_rope_fp8_quant_kernel(
    const uint16_t* __restrict__ o, const int64_t* __restrict__ positions,
    const float* __restrict__ cache, int64_t T, int64_t max_pos, int H, int hpg,
    uint8_t* __restrict__ out_fp8, int32_t* __restrict__ out_scale, int64_t T_al,
    int* __restrict__ status) {
  griddep_launch_dependents();  // a following GEMM may start its prologue now
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t groups = T * (H / kU);  // (token, kU-head group) work items
  const int64_t D = static_cast<int64_t>(hpg) * kHeadDim;
  const bool rope_lane = lane >= 24;
  const int quad = lane - 24;  // lanes 24-31: rope pairs 4*quad .. 4*quad+3

  for (int64_t item = warp; item < groups; item += nwarps) {
    const int64_t t = item / (H / kU);
    const int h0 = static_cast<int>(item - t * (H / kU)) * kU;
    const uint4* src = reinterpret_cast<const uint4*>(o + (t * H + h0) * kHeadDim);
    uint4 v0[kU], v1[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      v0[u] = __ldcs(src + u * (kHeadDim / 8) + lane);
      v1[u] = __ldcs(src + u * (kHeadDim / 8) + 32 + lane);
    }
    float4 c = make_float4(1.f, 1.f, 1.f, 1.f), sn = make_float4(0.f, 0.f, 0.f, 0.f);
    bool rotate = false;
    if (rope_lane) {
      const int64_t pos = __ldg(positions + t);
      if (pos >= 0 && pos < max_pos) {
        const float4* row = reinterpret_cast<const float4*>(cache + pos * kRope);
        c = __ldg(row + quad);
        sn = __ldg(row + 8 + quad);
        rotate = true;
      } else {
        record_status(status, DSV4_ERR_RANGE);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float f0[8], f1[8];
      unpack8(v0[u], f0);
      unpack8(v1[u], f1);
      if (rotate) {
        inv_rotate(f1[0], f1[1], c.x, sn.x);
        inv_rotate(f1[2], f1[3], c.y, sn.y);
        inv_rotate(f1[4], f1[5], c.z, sn.z);
        inv_rotate(f1[6], f1[7], c.w, sn.w);
      }
      float m0 = 0.f, m1 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m0 = fmaxf(m0, fabsf(f0[j]));
        m1 = fmaxf(m1, fabsf(f1[j]));
      }
      m0 = half_warp_max(m0);
      m1 = half_warp_max(m1);
      const int e0 = ue8m0_exponent(m0);
      const int e1 = ue8m0_exponent(m1);
      const uint2 q0 = quant8(f0, exp2_neg(e0));
      const uint2 q1 = quant8(f1, exp2_neg(e1));

      const int h = h0 + u;
      const int g = h / hpg;
      const int hh = h - g * hpg;
      uint8_t* dst = out_fp8 + (static_cast<int64_t>(g) * T + t) * D +
                     static_cast<int64_t>(hh) * kHeadDim;
      __stcs(reinterpret_cast<uint2*>(dst) + lane, q0);
      __stcs(reinterpret_cast<uint2*>(dst + 256) + lane, q1);

      // bytes: block 0 = e0 of lanes 0-15, block 1 = e0 of lanes 16-31,
      //        block 2 = e1 of lanes 0-15, block 3 = e1 of lanes 16-31
      const uint32_t b0 = static_cast<uint32_t>(e0 + 127);
      const uint32_t b2 = static_cast<uint32_t>(e1 + 127);
      const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, b0, 16);
      const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, b2, 16);
      if (lane == 0) {
        const uint32_t word = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
        out_scale[(static_cast<int64_t>(g) * hpg + hh) * T_al + t] = static_cast<int32_t>(word);
      }
    }
  }
}

// quantize=False: the same load / rotation, bf16 out in the group-major layout.
// Nope lanes are stored exactly as loaded; rotated lanes are rounded to bf16.
template <int kU>
__global__ void __launch_bounds__(256) inv_rope_bf16_kernel(
    const uint16_t* __restrict__ o, const int64_t* __restrict__ positions,
    const float* __restrict__ cache, int64_t T, int64_t max_pos, int H, int hpg,
    uint16_t* __restrict__ out, int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t groups = T * (H / kU);
  const int64_t D = static_cast<int64_t>(hpg) * kHeadDim;
  const bool rope_lane = lane >= 24;
  const int quad = lane - 24;
  for (int64_t item = warp; item < groups; item += nwarps) {
    const int64_t t = item / (H / kU);
    const int h0 = static_cast<int>(item - t * (H / kU)) * kU;
    const uint4* src = reinterpret_cast<const uint4*>(o + (t * H + h0) * kHeadDim);
    uint4 v0[kU], v1[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      v0[u] = __ldcs(src + u * (kHeadDim / 8) + lane);
      v1[u] = __ldcs(src + u * (kHeadDim / 8) + 32 + lane);
    }
    float4 c = make_float4(1.f, 1.f, 1.f, 1.f), sn = make_float4(0.f, 0.f, 0.f, 0.f);
    bool rotate = false;
    if (rope_lane) {
      const int64_t pos = __ldg(positions + t);
      if (pos >= 0 && pos < max_pos) {
        const float4* row = reinterpret_cast<const float4*>(cache + pos * kRope);
        c = __ldg(row + quad);
        sn = __ldg(row + 8 + quad);
        rotate = true;
      } else {
        record_status(status, DSV4_ERR_RANGE);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      uint4 w1 = v1[u];
      if (rotate) {
        float f1[8];
        unpack8(v1[u], f1);
        inv_rotate(f1[0], f1[1], c.x, sn.x);
        inv_rotate(f1[2], f1[3], c.y, sn.y);
        inv_rotate(f1[4], f1[5], c.z, sn.z);
        inv_rotate(f1[6], f1[7], c.w, sn.w);
        uint32_t wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(f1[2 * i], f1[2 * i + 1]);
          wv[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        w1 = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
      const int h = h0 + u;
      const int g = h / hpg;
      const int hh = h - g * hpg;
      uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<int64_t>(g) * T + t) * D +
                                            static_cast<int64_t>(hh) * kHeadDim);
      __stcs(dst + lane, v0[u]);
      __stcs(dst + 32 + lane, w1);
    }
  }
}

template <int kU>
void launch_bf16_u(const void* o, const int64_t* positions, const float* cache, int64_t T,
                   int64_t max_pos, int H, int hpg, void* out, cudaStream_t stream,
                   const DeviceInfo& dev) {
  const int threads = 256;
  const int64_t items = T * (H / kU);
  int64_t blocks = (items * 32 + threads - 1) / threads;
  // one wave: as many blocks as are resident at once (the registers bound it;
  // a second, partial wave of blocks measured 2-3 % slower)
  static std::atomic<int> resident[kMaxDevices];
  int per_sm = lazy_per_device(resident, dev.device, [&] {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, inv_rope_bf16_kernel<kU>, threads, 0) ==
                   cudaSuccess ? n : 0;
  });
  if (per_sm <= 0) per_sm = 2048 / threads;   // not known: a full SM's worth
  const int64_t max_blocks = static_cast<int64_t>(dev.num_sms) * per_sm;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  inv_rope_bf16_kernel<kU><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint16_t*>(o), positions, cache, T, max_pos, H, hpg,
      static_cast<uint16_t*>(out), dev.status);
}

template <int kU>
void launch_u(const void* o, const int64_t* positions, const float* cache, int64_t T,
              int64_t max_pos, int H, int hpg, void* out_fp8, int32_t* out_scale,
              cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t T_al = (T + 3) / 4 * 4;
  const int threads = 256;
  const int64_t items = T * (H / kU);
  int64_t blocks = (items * 32 + threads - 1) / threads;
  // one wave: as many blocks as are resident at once (the registers bound it;
  // a second, partial wave of blocks measured 2-3 % slower)
  static std::atomic<int> resident[kMaxDevices];
  int per_sm = lazy_per_device(resident, dev.device, [&] {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, inv_rope_fp8_quant_kernel<kU>, threads, 0) ==
                   cudaSuccess ? n : 0;
  });
  if (per_sm <= 0) per_sm = 2048 / threads;   // not known: a full SM's worth
  const int64_t max_blocks = static_cast<int64_t>(dev.num_sms) * per_sm;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  inv_rope_fp8_quant_kernel<kU><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint16_t*>(o), positions, cache, T, max_pos, H, hpg,
      static_cast<uint8_t*>(out_fp8), out_scale, T_al, dev.status);
}

}  // namespace

int launch_inv_rope_fp8_quant(const void* o, const int64_t* positions, const float* cache,
                              int64_t T, int64_t max_pos, int n_groups, int hpg,
                              void* out_fp8, int32_t* out_scale, cudaStream_t stream,
                              const DeviceInfo& dev) {
  const int H = n_groups * hpg;
  if (H % 4 == 0)
    launch_u<4>(o, positions, cache, T, max_pos, H, hpg, out_fp8, out_scale, stream, dev);
  else if (H % 2 == 0)
    launch_u<2>(o, positions, cache, T, max_pos, H, hpg, out_fp8, out_scale, stream, dev);
  else
    launch_u<1>(o, positions, cache, T, max_pos, H, hpg, out_fp8, out_scale, stream, dev);
  return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

int launch_inv_rope_bf16(const void* o, const int64_t* positions, const float* cache, int64_t T,
                         int64_t max_pos, int n_groups, int hpg, void* out, cudaStream_t stream,
                         const DeviceInfo& dev) {
  const int H = n_groups * hpg;
  if (H % 4 == 0)
    launch_bf16_u<4>(o, positions, cache, T, max_pos, H, hpg, out, stream, dev);
  else if (H % 2 == 0)
    launch_bf16_u<2>(o, positions, cache, T, max_pos, H, hpg, out, stream, dev);
  else
    launch_bf16_u<1>(o, positions, cache, T, max_pos, H, hpg, out, stream, dev);
  return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

}  // namespace dsv4
