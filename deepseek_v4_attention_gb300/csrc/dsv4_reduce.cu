// dsv4_reduce.cu -- the last step of group-split tensor parallelism: partial
// O-projection outputs (fp32, one per group range) summed and rounded to the
// bf16 output.  With one partial it is the conversion that follows an fp32
// reduce-scatter.  HBM-bound: 4 n + 2 bytes per output element.
#include <cuda_bf16.h>

#include "../../include/dsv4.h"
#include "dsv4_internal.h"

namespace dsv4 {

namespace {

struct Parts {
  const float* p[DSV4_MAX_PARTIALS];
};

// Each thread sums 8 consecutive elements of every partial (two 16-byte loads
// per partial), in the order 0, 1, ..., n-1, and writes 8 bf16 (one 16-byte
// store); the elems % 8 tail is taken element by element.
__global__ void __launch_bounds__(256) sum_partials_kernel(Parts parts, int n, int64_t elems,
                                                           uint16_t* out) {
  const int64_t n8 = elems / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += stride) {
    const float4* s0 = reinterpret_cast<const float4*>(parts.p[0]) + 2 * i;
    float4 a = __ldcs(s0), b = __ldcs(s0 + 1);
    for (int j = 1; j < n; ++j) {
      const float4* sj = reinterpret_cast<const float4*>(parts.p[j]) + 2 * i;
      const float4 c = __ldcs(sj), d = __ldcs(sj + 1);
      a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
      b.x += d.x; b.y += d.y; b.z += d.z; b.w += d.w;
    }
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y);
    const __nv_bfloat162 h1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(b.x, b.y);
    const __nv_bfloat162 h3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 v;
    v.x = *reinterpret_cast<const uint32_t*>(&h0);
    v.y = *reinterpret_cast<const uint32_t*>(&h1);
    v.z = *reinterpret_cast<const uint32_t*>(&h2);
    v.w = *reinterpret_cast<const uint32_t*>(&h3);
    __stcs(reinterpret_cast<uint4*>(out) + i, v);
  }
  for (int64_t e = 8 * n8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       e < elems; e += stride) {
    float acc = parts.p[0][e];
    for (int j = 1; j < n; ++j) acc += parts.p[j][e];
    const __nv_bfloat16 h = __float2bfloat16_rn(acc);
    out[e] = *reinterpret_cast<const uint16_t*>(&h);
  }
}

}  // namespace

int launch_sum_partials(const float* const* parts, int n, int64_t elems, void* out_bf16,
                        cudaStream_t stream, const DeviceInfo& dev) {
  Parts ps = {};
  for (int j = 0; j < n; ++j) ps.p[j] = parts[j];
  const int threads = 256;
  const int64_t work = (elems / 8 > 0 ? elems / 8 : elems);
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t wave = static_cast<int64_t>(dev.num_sms) * (2048 / threads);
  if (blocks > wave) blocks = wave;
  if (blocks < 1) blocks = 1;
  sum_partials_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      ps, n, elems, static_cast<uint16_t*>(out_bf16));
  return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

}  // namespace dsv4
