// dsv4_gemm_pair.cu -- the block-scaled FP8 GEMM on CTA pairs
// (tcgen05.mma.cta_group::2), for the large shapes of both projections (the
// grouped wo_a with its fused z re-quantisation, the dense wo_b), and its
// bf16 form (kBf16: kind::f16, no scale factors) for the non-FP8 grouped wo_a:
//
//   C[t, g*N + n] = sum_k A[g][t][k] 2^ea[g][t][k/128] * B[g*N+n][k] 2^eb[(g*N+n)/128][k/128]
//
// A cluster of two CTAs (on two SMs) computes a 256-token x 256-column tile.
// Each CTA stages its own 128 token rows of A and its own 128 of the tile's
// B rows (output columns); one thread of the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 32; K = 16 bf16), which reads both CTAs'
// shared memory and leaves in each CTA's tensor memory the 128 x 256 fp32
// accumulator of its own tokens.  Per SM and 128-deep k-block the operands are
// 32 KiB (48 KiB for a 128 x 256 tile on one SM), so the same shared memory
// holds six k-blocks instead of four.  They form three stages of two k-blocks
// (eight MMAs) each: the MMA thread waits once and commits once per eight
// MMAs (a wait per four measured ~0.7 of the ideal issue rate even with the
// operands resident, a wait per eight 1.0), and a stage's refill still has
// two stages of MMAs (2048 cycles) to land in.
//
// Roles (both CTAs unless said otherwise):
//   warp 0, lane 0   producer: its A and B halves of each stage's k-blocks, by
//                    TMA; the copies complete on the even CTA's full barrier
//                    (which expects the bytes of both CTAs).
//   warp 1, lane 0   (even CTA) MMA issuer: at the first k-block of each pack
//                    of four, tcgen05.cp of the stage's scale factors into a
//                    TMEM region of both CTAs; per k-block four MMAs, per
//                    stage one commit that frees it in both CTAs (multicast).
//   warp 2           (FP8) scale factors: at the first k-block of a pack each CTA
//                    writes the 128 A scale words of its own tokens and the B
//                    scales of all 256 columns into the stage's slot of its own
//                    shared memory.  The even CTA's warp then arrives on the
//                    stage's full barrier; the odd CTA's warp signals its slot
//                    with a 16-byte bulk copy into the even CTA's shared memory
//                    whose completion counts as transaction bytes on that same
//                    barrier (an arrive at cluster scope costs ~2000 cycles, a
//                    bulk copy's completion rides the TMA path).
//   warps 3..10      epilogue: the CTA's 128 x 256 accumulator to registers
//                    (each warp 32 rows x 128 columns, one tcgen05.ld), a
//                    release of the accumulator to the even CTA's MMA thread
//                    (the odd CTA's warps: a 16-byte bulk copy into the even
//                    CTA's shared memory, counted as transaction bytes on its
//                    barrier), then the bf16 /
//                    fp32 store or the per-128 FP8 re-quantisation, through a
//                    swizzled staging buffer and TMA stores.
// Every wait is bounded (the library's 2 s limit); a timeout records
// DSV4_ERR_TIMEOUT, every role of the CTA leaves its loop, and both CTAs meet
// at the final cluster barrier before the tensor memory is released.
#include "dsv4_gemm_common.cuh"

namespace dsv4 {

namespace {

// ------------------------------------------------ CTA pairs (cta_group::2) --
// Allocation and release of tensor memory are done by one warp of each CTA;
// every tcgen05 instruction of the kernel uses .cta_group::2.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem,
                                              uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on the mbarrier at the same shared-memory offset in both CTAs of the
// pair once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Arrives on this CTA's mbarrier once every tcgen05 operation issued so far by
// this thread is done.
__device__ __forceinline__ void mma_commit_own(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Shared memory -> tensor memory of both CTAs, each from its own shared
// memory at the same offset (32 rows of 16 bytes, broadcast to the four
// 32-lane quarters).
__device__ __forceinline__ void tmem_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// TMA loads into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of the pair (`bar_cluster`: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y,
                                                 int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory into
// another CTA's (dst_cluster, a shared::cluster address); its completion is
// counted as transaction bytes on that CTA's mbarrier bar_cluster.
__device__ __forceinline__ void bulk_copy_to_cta(uint32_t dst_cluster, const void* src,
                                                 uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
      " [%0], [%1], %2, [%3];" ::"r"(dst_cluster),
      "r"(smem_addr(src)), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

// Each thread of the warp reads 128 consecutive 32-bit columns of its own lane
// (one instruction instead of four 32-column loads: fewer registers live in
// the re-quantising epilogue, no spills).
__device__ __forceinline__ void tmem_ld_128cols(uint32_t taddr, uint32_t (&r)[4][32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];"
      : "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]), "=r"(r[0][6]), "=r"(r[0][7]), "=r"(r[0][8]), "=r"(r[0][9]), "=r"(r[0][10]), "=r"(r[0][11]), "=r"(r[0][12]), "=r"(r[0][13]), "=r"(r[0][14]), "=r"(r[0][15]), "=r"(r[0][16]), "=r"(r[0][17]), "=r"(r[0][18]), "=r"(r[0][19]), "=r"(r[0][20]), "=r"(r[0][21]), "=r"(r[0][22]), "=r"(r[0][23]), "=r"(r[0][24]), "=r"(r[0][25]), "=r"(r[0][26]), "=r"(r[0][27]), "=r"(r[0][28]), "=r"(r[0][29]), "=r"(r[0][30]), "=r"(r[0][31]), "=r"(r[1][0]), "=r"(r[1][1]), "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]), "=r"(r[1][6]), "=r"(r[1][7]), "=r"(r[1][8]), "=r"(r[1][9]), "=r"(r[1][10]), "=r"(r[1][11]), "=r"(r[1][12]), "=r"(r[1][13]), "=r"(r[1][14]), "=r"(r[1][15]), "=r"(r[1][16]), "=r"(r[1][17]), "=r"(r[1][18]), "=r"(r[1][19]), "=r"(r[1][20]), "=r"(r[1][21]), "=r"(r[1][22]), "=r"(r[1][23]), "=r"(r[1][24]), "=r"(r[1][25]), "=r"(r[1][26]), "=r"(r[1][27]), "=r"(r[1][28]), "=r"(r[1][29]), "=r"(r[1][30]), "=r"(r[1][31]), "=r"(r[2][0]), "=r"(r[2][1]), "=r"(r[2][2]), "=r"(r[2][3]), "=r"(r[2][4]), "=r"(r[2][5]), "=r"(r[2][6]), "=r"(r[2][7]), "=r"(r[2][8]), "=r"(r[2][9]), "=r"(r[2][10]), "=r"(r[2][11]), "=r"(r[2][12]), "=r"(r[2][13]), "=r"(r[2][14]), "=r"(r[2][15]), "=r"(r[2][16]), "=r"(r[2][17]), "=r"(r[2][18]), "=r"(r[2][19]), "=r"(r[2][20]), "=r"(r[2][21]), "=r"(r[2][22]), "=r"(r[2][23]), "=r"(r[2][24]), "=r"(r[2][25]), "=r"(r[2][26]), "=r"(r[2][27]), "=r"(r[2][28]), "=r"(r[2][29]), "=r"(r[2][30]), "=r"(r[2][31]), "=r"(r[3][0]), "=r"(r[3][1]), "=r"(r[3][2]), "=r"(r[3][3]), "=r"(r[3][4]), "=r"(r[3][5]), "=r"(r[3][6]), "=r"(r[3][7]), "=r"(r[3][8]), "=r"(r[3][9]), "=r"(r[3][10]), "=r"(r[3][11]), "=r"(r[3][12]), "=r"(r[3][13]), "=r"(r[3][14]), "=r"(r[3][15]), "=r"(r[3][16]), "=r"(r[3][17]), "=r"(r[3][18]), "=r"(r[3][19]), "=r"(r[3][20]), "=r"(r[3][21]), "=r"(r[3][22]), "=r"(r[3][23]), "=r"(r[3][24]), "=r"(r[3][25]), "=r"(r[3][26]), "=r"(r[3][27]), "=r"(r[3][28]), "=r"(r[3][29]), "=r"(r[3][30]), "=r"(r[3][31])
      : "r"(taddr)
      : "memory");
}

constexpr int kPairM = 2 * kBM;   // tokens per pair tile
constexpr int kPairRasterM = kRasterM / 2;

struct PairCfg {
  static constexpr int kBN = 256;                        // output columns per pair tile
  static constexpr uint32_t kABytes = kBM * kBK;         // this CTA's 128 token rows
  static constexpr uint32_t kBBytes = (kBN / 2) * kBK;   // this CTA's 128 output columns
  static constexpr int kSlots = 6;                       // k-block buffers
  static constexpr int kKps = 2;                         // k-blocks per stage
  static constexpr int kStages = kSlots / kKps;
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiWarp0 = 3;
  static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
  static constexpr uint32_t kSfbBytes = kBN * 4;         // the scales of all 256 columns
  static constexpr uint32_t kSfSlotBytes = kSfaBytes + kSfbBytes;
  static constexpr int kSfCol0 = kBN;                    // TMEM: after the accumulator
  static constexpr int kSfColsPerSlot = 4 + kBN / 32;
  static_assert(kSfCol0 + kStages * kSfColsPerSlot <= kTmemCols, "TMEM budget");
  static constexpr uint32_t a = 0;
  static constexpr uint32_t b = a + kSlots * kABytes;
  static constexpr uint32_t sf = b + kSlots * kBBytes;
  static constexpr uint32_t kEpiBufBytes = 2048;
  static constexpr uint32_t epi = (sf + kStages * kSfSlotBytes + 1023) / 1024 * 1024;
  static constexpr uint32_t bars = epi + kEpiWarps * kEpiBufBytes;
  // full/empty[kStages], tmem_full, tmem_empty, drain
  static constexpr uint32_t n_bars = 2 * kStages + 3;
  static constexpr uint32_t misc = bars + n_bars * 8;    // tmem base, abort flag
  // 16 bytes per stage that the odd CTA's slot signal lands on (even CTA)
  static constexpr uint32_t sig = (misc + 16 + 15) / 16 * 16;
  // 16 bytes per epilogue warp that the odd CTA's accumulator release lands on
  static constexpr uint32_t esig = sig + 16 * kStages;
  static constexpr uint32_t total = esig + 16 * kEpiWarps;
  static constexpr uint32_t smem_bytes = total + 1024;   // + alignment slack
};

// kBf16: A and B bf16 (a k-block is 64 elements, still 128 bytes a row),
// tcgen05.mma.kind::f16 without scale factors, bf16 output only.
template <int kEpi, bool kBf16>
__global__ void __launch_bounds__(PairCfg::kThreads, 1)
    block_scaled_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a,
                                  const __grid_constant__ CUtensorMap tm_b,
                                  const __grid_constant__ CUtensorMap tm_out, const Params p) {
  using C = PairCfg;
  static_assert(!kBf16 || kEpi == kEpiBf16, "the bf16 GEMM has the bf16 epilogue only");
  constexpr int kStages = C::kStages;
  constexpr int kKps = C::kKps;
  constexpr int kBKe = kBf16 ? 64 : kBK;   // elements of K per 128-byte k-block
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bars);
  uint64_t* full = bars;                 // used in the even CTA
  uint64_t* empty = full + kStages;      // both CTAs (multicast commits)
  uint64_t* tmem_full = empty + kStages; // both CTAs (multicast commit)
  uint64_t* tmem_empty = tmem_full + 1;  // the even CTA's: both CTAs' epilogue warps arrive
  uint64_t* drain = tmem_empty + 1;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + C::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();
  const uint32_t rank = cluster_cta_rank();   // 0: the CTA that issues the MMAs
  const bool leader = rank == 0;
  const int pair0 = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // the producer's expect_tx and (FP8) the scale-factor warp
      mbar_init(&full[s], kBf16 ? 1 : 2);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, C::kEpiWarps);   // the even CTA's warps; the odd's by transaction bytes
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_base_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_slot;
  griddep_wait();   // every operand may come from the previous kernel

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint32_t full_leader = map_to_cta(smem_addr(full), 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair0; tile < p.num_tiles && ok; tile += npairs) {
        int g, n_blk, m_blk;
        tile_coords(p, tile, g, n_blk, m_blk);
        const int m0 = m_blk * kPairM + static_cast<int>(rank) * kBM;
        const int brow = g * p.N + n_blk * C::kBN + static_cast<int>(rank) * (C::kBN / 2);
        for (int kbs = 0; kbs < p.k_blocks; kbs += kKps) {
          const int n = p.k_blocks - kbs >= kKps ? kKps : p.k_blocks - kbs;
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          // the even CTA's barrier expects both CTAs' operands and, when the
          // stage starts a pack, the odd CTA's 16-byte slot signal
          if (leader)
            mbar_arrive_expect_tx(&full[stage],
                                  2u * static_cast<uint32_t>(n) * (C::kABytes + C::kBBytes) +
                                      ((!kBf16 && (kbs & 3) == 0) ? 16u : 0u));
          const uint32_t fb = full_leader + 8u * static_cast<uint32_t>(stage);
          for (int j = 0; j < n; ++j) {
            const int slot = stage * kKps + j;
            tma_load_3d_pair(smem + C::a + slot * C::kABytes, &tm_a, fb, (kbs + j) * kBKe, m0, g);
            tma_load_2d_pair(smem + C::b + slot * C::kBBytes, &tm_b, fb, (kbs + j) * kBKe, brow);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // Copies in flight complete on the even CTA's barriers, which this
        // thread cannot wait on: give them time to land (both CTAs stay
        // resident until the final cluster barrier).
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------- MMA issue
      const uint64_t adesc0 = smem_desc(smem_addr(smem + C::a), 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_addr(smem + C::b), 16, 1024, 2);
      const uint64_t sfdesc0 = smem_desc(smem_addr(smem + C::sf), 0, 128, 0);
      const uint32_t idesc0 = kBf16 ? bf16_idesc(kPairM, C::kBN) : mxf8_idesc(kPairM, C::kBN, 0, 0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      // A pack's scale words serve its four k-blocks (the scale-factor id
      // picks the byte): copied to TMEM once per pack, into region (packs so
      // far) mod kStages, rewritten kStages packs later, when the stage's
      // full-barrier wait proves every MMA at least kStages stages back done.
      // Stages start at even k-blocks, so only a stage's first k-block can
      // start a pack.
      int sf_region = kStages - 1;
      uint32_t sf_col = 0;
      bool ok = true;
      for (int tile = pair0; tile < p.num_tiles && ok; tile += npairs) {
        // the accumulator is free once both CTAs' epilogues have read it
        if (!mbar_wait(tmem_empty, acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        for (int kbs = 0; kbs < p.k_blocks; kbs += kKps) {
          const int n = p.k_blocks - kbs >= kKps ? kKps : p.k_blocks - kbs;
          // both CTAs' operands, both scale-factor slots at a pack start
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          if (!kBf16 && (kbs & 3) == 0) {
            sf_region = (sf_region + 1 == kStages) ? 0 : sf_region + 1;
            sf_col = tmem_base + static_cast<uint32_t>(C::kSfCol0 + sf_region * C::kSfColsPerSlot);
            const uint64_t sd = sfdesc0 + ((stage * C::kSfSlotBytes) >> 4);
            tmem_cp_32x128b_x4_pair(sf_col, sd);                 // A: 512 B
#pragma unroll
            for (int r = 0; r < C::kBN / 128; ++r)               // B: 512 B per 128 columns
              tmem_cp_32x128b_x4_pair(sf_col + 4 + 4 * r, sd + ((kSfaBytes + 512u * r) >> 4));
          }
#pragma unroll
          for (int j = 0; j < kKps; ++j) {
            if (j < n) {
              const int kb = kbs + j;
              const int slot = stage * kKps + j;
              const uint64_t ad = adesc0 + ((slot * C::kABytes) >> 4);
              const uint64_t bd = bdesc0 + ((slot * C::kBBytes) >> 4);
              const uint32_t sfid = kBf16 ? 0u : static_cast<uint32_t>(kb & 3);
              const uint32_t id = idesc0 | (sfid << 4) | (sfid << 29);
              // four MMAs per k-block: K = 32 e4m3 or K = 16 bf16, 32 bytes each
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if constexpr (kBf16)
                  mma_bf16_pair(tmem_base, ad + 2 * k, bd + 2 * k, id, (kb | k) != 0 ? 1u : 0u);
                else
                  mma_mxf8_pair(tmem_base, ad + 2 * k, bd + 2 * k, id, sf_col, sf_col + 4,
                                (kb | k) != 0 ? 1u : 0u);
              }
            }
          }
          mma_commit_both(&empty[stage]);   // frees the stage in both CTAs
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_both(tmem_full);
        acc_phase ^= 1u;
      }
      if (*abort_flag) {
        // every MMA and copy issued here completes before TMEM is released
        mma_commit_own(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else if (warp == 2 && !kBf16) {
    // ------------------------------------------------------ scale factors
    constexpr int kRb = C::kBN / 128;   // 128-column weight-scale blocks per tile
    const int packs = p.packs;
    const uint32_t full_leader = map_to_cta(smem_addr(full), 0);
    const uint32_t sig_leader = map_to_cta(smem_addr(smem + C::sig), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = pair0; tile < p.num_tiles && ok; tile += npairs) {
      int g, n_blk, m_blk;
      tile_coords(p, tile, g, n_blk, m_blk);
      const int rb = (g * p.N + n_blk * C::kBN) / 128;
      // the tile's weight-scale words: lane l holds packs l, l + 32, ...
      uint32_t wcur[kRb][4];
#pragma unroll
      for (int r = 0; r < kRb; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          wcur[r][i] = (lane + 32 * i < packs) ? b_scale_word(p, rb + r, lane + 32 * i) : 0u;
      // this CTA's 128 tokens; lane l takes rows l, l + 32, l + 64, l + 96
      const int64_t m0 = static_cast<int64_t>(m_blk) * kPairM + static_cast<int64_t>(rank) * kBM;
      for (int kbs = 0; kbs < p.k_blocks; kbs += kKps) {
        const bool pack_start = (kbs & 3) == 0;
        uint32_t va[4] = {0u, 0u, 0u, 0u}, bword[kRb];
        if (pack_start) {
          const int j = kbs / 4;
          const int32_t* src = p.a_scale + (static_cast<int64_t>(g) * packs + j) * p.t_al;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int64_t t = m0 + 32 * c + lane;
            va[c] = (t < p.T) ? static_cast<uint32_t>(__ldg(src + t)) : 0u;
          }
#pragma unroll
          for (int r = 0; r < kRb; ++r) {
            const uint32_t src_w = (j < 32) ? wcur[r][0] : (j < 64) ? wcur[r][1]
                                 : (j < 96) ? wcur[r][2] : wcur[r][3];
            bword[r] = __shfl_sync(0xFFFFFFFFu, src_w, j & 31);
          }
        }
        // the slot is free once the stage's MMAs and copies are done
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (pack_start) {
          uint4* dst = reinterpret_cast<uint4*>(smem + C::sf + stage * C::kSfSlotBytes);
          dst[lane] = make_uint4(va[0], va[1], va[2], va[3]);
#pragma unroll
          for (int r = 0; r < kRb; ++r)
            dst[32 + 32 * r + lane] = make_uint4(bword[r], bword[r], bword[r], bword[r]);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          if (leader) {
            mbar_arrive(&full[stage]);
          } else if (pack_start) {
            bulk_copy_to_cta(sig_leader + 16u * static_cast<uint32_t>(stage),
                             smem + C::sf + stage * C::kSfSlotBytes, 16u,
                             full_leader + 8u * static_cast<uint32_t>(stage));
          }
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && !leader) {
      // a slot signal in flight completes on the even CTA's barrier: give it
      // time to land (both CTAs stay resident until the final cluster barrier)
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 1000000ull) {
      }
    }
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int epi = warp - C::kEpiWarp0;  // 0 .. 7
    const int quarter = warp & 3;         // TMEM lanes this warp may access
    const int col_half = epi >> 2;        // which 128 columns of the tile
    const int row = quarter * 32 + lane;
    const uint32_t tmem_empty_leader = map_to_cta(smem_addr(tmem_empty), 0);
    const uint32_t esig_leader = map_to_cta(smem_addr(smem + C::esig), 0);
    uint32_t acc_phase = 0;
    for (int tile = pair0; tile < p.num_tiles; tile += npairs) {
      int g, n_blk, m_blk;
      tile_coords(p, tile, g, n_blk, m_blk);
      if (!mbar_wait_warp(tmem_full, acc_phase, abort_flag, p.status)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      const int64_t m0 = static_cast<int64_t>(m_blk) * kPairM + static_cast<int64_t>(rank) * kBM;
      const int64_t t = m0 + row;
      const bool live = t < p.T;
      const int64_t col0 = static_cast<int64_t>(g) * p.N + static_cast<int64_t>(n_blk) * C::kBN +
                           128 * col_half;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(128 * col_half);
      uint32_t r[4][32];
      tmem_ld_128cols(taddr, r);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      // The accumulator may be overwritten once all 16 warps have read it: the
      // even CTA's eight arrive (its warp 0 expecting the odd CTA's 8 x 16
      // bytes), the odd CTA's send 16 bytes each into the even CTA's shared
      // memory, completing on the same barrier.  Nothing is sent after the
      // pair's last tile (no MMA waits for it; no copy may be in flight when
      // the CTAs exit).
      if (lane == 0) {
        const bool more = tile + npairs < p.num_tiles;
        if (leader) {
          if (epi == 0 && more) mbar_arrive_expect_tx(tmem_empty, 16u * C::kEpiWarps);
          else mbar_arrive(tmem_empty);
        } else if (more) {
          bulk_copy_to_cta(esig_leader + 16u * static_cast<uint32_t>(epi),
                           smem + C::esig + 16 * epi, 16u, tmem_empty_leader);
        }
      }
      // Stores through this warp's staging buffer: each lane writes its row's
      // 64-byte chunk with the 64-byte TMA swizzle (16-byte unit q of row r at
      // q ^ ((r >> 1) & 3)), then one lane stores the 32-row box with TMA,
      // which also clips rows beyond T.
      uint8_t* buf = smem + C::epi + epi * C::kEpiBufBytes;
      const int32_t box_y = static_cast<int32_t>(m0 + quarter * 32);
      auto stage_chunk = [&](const uint4 (&v)[4], int32_t box_x) {
        if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(buf + 64 * lane + 16 * (q ^ ((lane >> 1) & 3))) = v[q];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && box_y < p.T) {   // a box wholly past the last row is skipped
          tma_store_2d(&tm_out, buf, box_x, box_y);
          bulk_commit_group();
        }
      };
      if constexpr (kEpi == kEpiF32) {
        // eight chunks of 16 columns (64 bytes of fp32 per row)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int bcol = 16 * (c & 1) + 4 * q;
            v[q] = make_uint4(r[c >> 1][bcol], r[c >> 1][bcol + 1], r[c >> 1][bcol + 2],
                              r[c >> 1][bcol + 3]);
          }
          stage_chunk(v, static_cast<int32_t>(col0 + 16 * c));
        }
      } else if constexpr (kEpi == kEpiBf16) {
        // four chunks of 32 columns (64 bytes of bf16 per row)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __nv_bfloat162 h = __floats2bfloat162_rn(
                  __uint_as_float(r[c][8 * q + 2 * i]), __uint_as_float(r[c][8 * q + 2 * i + 1]));
              w[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
            v[q] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          stage_chunk(v, static_cast<int32_t>(col0 + 32 * c));
        }
      } else {
        // z is a bf16 tensor: round first, then quantise the rounded values
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float zr = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[c][i])));
            r[c][i] = __float_as_uint(zr);
            amax = fmaxf(amax, fabsf(zr));
          }
        const int e = ue8m0_exponent(amax);
        const float inv = exp2_neg(e);
        // two chunks of 64 columns (64 bytes of e4m3 per row)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c = 2 * h + (q >> 1);
              const int bcol = 16 * (q & 1) + 4 * i;
              w[i] = static_cast<uint32_t>(e4m3x2(__uint_as_float(r[c][bcol]) * inv,
                                                  __uint_as_float(r[c][bcol + 1]) * inv)) |
                     (static_cast<uint32_t>(e4m3x2(__uint_as_float(r[c][bcol + 2]) * inv,
                                                   __uint_as_float(r[c][bcol + 3]) * inv))
                      << 16);
            }
            v[q] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          stage_chunk(v, static_cast<int32_t>(col0 + 64 * h));
        }
        if (live) {
          const int64_t blk = col0 / 128;  // 128-column block of the flattened row
          uint8_t* sbytes = reinterpret_cast<uint8_t*>(p.q_scale);
          sbytes[((blk >> 2) * p.t_al + t) * 4 + (blk & 3)] = static_cast<uint8_t>(e + 127);
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // every store complete before the CTA leaves
    __syncwarp();
    if (!leader && *abort_flag && lane == 0) {
      // a release signal in flight completes on the even CTA's barrier: give
      // it time to land (both CTAs stay resident until the final barrier)
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 1000000ull) {
      }
    }
    __syncwarp();
  }

  // Both CTAs stay until neither can touch the other's shared memory, barriers
  // or tensor memory any more; then each releases its tensor memory.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int kEpi, bool kBf16 = false>
int launch_pair(const GemmProblem& q, cudaStream_t stream, const DeviceInfo& dev) {
  using C = PairCfg;
  static std::atomic<int> configured_for[kMaxDevices];
  if (dev.device < 0 || dev.device >= kMaxDevices) return DSV4_ERR_UNSUPPORTED;
  const int configured = lazy_per_device(configured_for, dev.device, [] {
    return cudaFuncSetAttribute(block_scaled_gemm_pair_kernel<kEpi, kBf16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::smem_bytes)) == cudaSuccess ? 1 : 0;
  });
  if (!configured) return DSV4_ERR_CUDA;
  const int64_t T = q.T;
  const int64_t t_al = (T + 3) / 4 * 4;
  // operands: 128-byte rows of K per k-block (128 e4m3 or 64 bf16 elements)
  const int esz = kBf16 ? 2 : 1;
  const int kbe = kBK / esz;
  const CUtensorMapDataType dt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap tm_a, tm_b, tm_out;
  {
    // A: [G][T][K]; a box is this CTA's 128 token rows x one 128-byte k-block
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(q.K), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(q.G)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(q.K) * esz,
                             static_cast<cuuint64_t>(T * q.K) * esz};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kbe), static_cast<cuuint32_t>(kBM), 1};
    if (!encode(&tm_a, dt, 3, q.a, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return DSV4_ERR_CUDA;
  }
  {
    // B: [G*N][K]; a box is this CTA's 128 output columns x one k-block
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(q.K),
                          static_cast<cuuint64_t>(static_cast<int64_t>(q.G) * q.N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(q.K) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kbe), static_cast<cuuint32_t>(C::kBN / 2)};
    if (!encode(&tm_b, dt, 2, q.b, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return DSV4_ERR_CUDA;
  }
  {
    // rows of G*N elements; a box is 32 rows x 64 bytes
    const int64_t ld = static_cast<int64_t>(q.G) * q.N;
    const int osz = kEpi == kEpiQuant ? 1 : kEpi == kEpiF32 ? 4 : 2;
    const void* base = kEpi == kEpiQuant ? static_cast<const void*>(q.q_out)
                       : kEpi == kEpiF32 ? static_cast<const void*>(q.out_f32)
                                         : q.out_bf16;
    const CUtensorMapDataType odt = kEpi == kEpiQuant ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                    : kEpi == kEpiF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(ld), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * osz)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / osz), 32u};
    if (!encode(&tm_out, odt, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return DSV4_ERR_CUDA;
  }
  Params p = {};
  p.T = T;
  p.G = q.G;
  p.N = q.N;
  p.K = q.K;
  p.m_tiles = static_cast<int>((T + kPairM - 1) / kPairM);   // 256-token blocks
  p.n_tiles = q.N / C::kBN;
  p.num_tiles = p.m_tiles * p.n_tiles * q.G;
  p.k_blocks = q.K / kbe;
  p.packs = (q.K / 128 + 3) / 4;
  p.t_al = t_al;
  p.a_scale = q.a_scale;
  p.b_scale = q.b_scale;
  p.b_scale_ld = q.K / 128;
  p.out = static_cast<__nv_bfloat16*>(q.out_bf16);
  p.q_out = q.q_out;
  p.q_scale = q.q_scale;
  p.status = dev.status;
  p.raster_m = (q.G == 1 && p.m_tiles > kPairRasterM) ? kPairRasterM : 0;
  p.prefetch_l2 = 0;

  // Persistent pairs, as many as can be resident at once (one CTA per SM; a
  // pair needs two SMs of one GPC, so an SM may be left over): a pair that
  // had to wait for a second wave would hold its share of the tiles back.
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = 2;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  static std::atomic<int> resident_pairs[kMaxDevices];
  const int max_pairs = lazy_per_device(resident_pairs, dev.device, [&] {
    cudaLaunchConfig_t c = cfg;
    c.gridDim = dim3(static_cast<unsigned>(2 * (dev.num_sms / 2)));
    c.attrs = attr;
    c.numAttrs = 1;
    int n = 0;
    return cudaOccupancyMaxActiveClusters(&n, block_scaled_gemm_pair_kernel<kEpi, kBf16>, &c) ==
                   cudaSuccess ? n : 0;
  });
  if (max_pairs <= 0) return DSV4_ERR_CUDA;
  const int pairs = p.num_tiles < max_pairs ? p.num_tiles : max_pairs;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  if (q.after_own_kernel) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, block_scaled_gemm_pair_kernel<kEpi, kBf16>, tm_a, tm_b, tm_out, p) !=
      cudaSuccess)
    return DSV4_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

}  // namespace

bool pair_gemm_eligible(const GemmProblem& q, const DeviceInfo& dev) {
  if (q.fused_a || q.N % PairCfg::kBN != 0) return false;
  if (q.bf16) {
    if (q.K % 64 != 0 || q.epilogue != kEpiBf16) return false;
  } else {
    if (q.K % kBK != 0 || q.K / 128 > 4 * 32 * 4) return false;   // weight-scale words per lane
  }
  const int64_t pair_tiles = (q.T + kPairM - 1) / kPairM * (q.N / PairCfg::kBN) * q.G;
  return q.T > kBM && pair_tiles >= dev.num_sms / 2;
}

int launch_pair_gemm(const GemmProblem& q, cudaStream_t stream, const DeviceInfo& dev) {
  if (q.bf16) return launch_pair<kEpiBf16, true>(q, stream, dev);
  switch (q.epilogue) {
    case kEpiQuant: return launch_pair<kEpiQuant>(q, stream, dev);
    case kEpiF32: return launch_pair<kEpiF32>(q, stream, dev);
    default: return launch_pair<kEpiBf16>(q, stream, dev);
  }
}

}  // namespace dsv4
