// dsv4_gemm.cu -- block-scaled FP8 GEMM on the 5th-generation tensor cores
// (tcgen05, kind::mxf8f6f4 with UE8M0 block scales), for both projections of
// the O-projection:
//   - grouped wo_a (vLLM docs, grouped_wo_a: group g meets rows g*R:(g+1)*R;
//     o_proj page, fp8_einsum("bhr,hdr->bhd") with recipe (1, 1, 128)),
//   - dense wo_b over z.flatten(1) (the same kernel with G = 1).
//
//   C[t, g*N + n] = sum_k A[g][t][k] 2^ea[g][t][k/128] * B[g*N+n][k] 2^eb[(g*N+n)/128][k/128]
//
// This file holds the one-SM kernel, used for the shapes the CTA-pair kernel
// (dsv4_gemm_pair.cu: 256 x 256 tiles on two SMs, the large FP8 shapes) does
// not take: decode and mid sizes, the bf16 path, the quantiser-fused decode
// kernel.  launch_block_scaled_gemm() below picks the kernel.
//
// Persistent, warp-specialised CTA, one per SM, tile 128 x kBN x 128 (kBN = 128
// or 256, see Cfg):
//   warp 0, lane 0   TMA producer: A tile (128 tokens x 128 k) and B tile
//                    (kBN rows x 128 k), both with the 128-byte swizzle.
//   warp 1, lane 0   MMA issuer: at the first k-block of each pack of four,
//                    tcgen05.cp of the stage's scale factors into a TMEM
//                    region; per k-block four tcgen05.mma (K = 32) from
//                    precomputed descriptors; per stage (one or two k-blocks,
//                    see Cfg) one commit that frees it.
//   warp 2           scale-factor warp: each stage has its own scale-factor
//                    slot, filled for the stage's k-block and completed on the
//                    stage's full barrier (which therefore counts two
//                    arrivals: the producer's and this warp's).  It loads the
//                    A scale words of a pack (one packed int32 per row) with
//                    coalesced loads, one pack ahead, and stores them in the
//                    32 x 16-byte order tcgen05.cp.32x128b.warpx4 expects
//                    (TMEM column c of lane r = row 32 c + r); it expands the
//                    raw 128 x 128 UE8M0 weight bytes into the kBN-row B
//                    scales.  The stage's empty barrier (committed after the
//                    MMAs that read the stage) guards the slot.
//   warps 3..        epilogue: per warp a 32-row x 128-column slice of the fp32
//                    accumulator to registers (tcgen05.ld), release of the
//                    accumulator, then bf16 conversion or the fused per-128
//                    FP8 re-quantisation (one thread holds one whole 128-block);
//                    the results leave through a swizzled shared-memory box
//                    and a TMA store (coalesced, rows beyond T clipped).
//   fused A (kFused, decode sizes): the TMA thread loads, instead of the FP8 A
//                    tile, the k-block's bf16 slice of the attention output
//                    into a small ring; four producer warps after the
//                    epilogue warps apply the quantiser's arithmetic to it
//                    and write the FP8 A tile and its scale bytes into the
//                    stage (the stage's full barrier then counts six
//                    arrivals).
// The producer and the MMA issuer are single-thread loops: their per-k-block
// instruction chain is what feeds the tensor pipe.
//
// Scale factors and the K = 128 blocks: the hardware applies one UE8M0 scale
// per 32 k (scale_vec::1X).  A 128-wide k-block is issued as four K = 32 MMAs
// that all select the same scale byte, which is exact: the four products are
// scaled by the same power of two.  The byte is chosen with the
// scale-factor-id field of the instruction descriptor: the 4 blocks of a
// packed int32 are bytes 0..3 of one TMEM column word.
#include "dsv4_gemm_common.cuh"

namespace dsv4 {

namespace {

// Tile configuration.  kBN = 128: two 128-column TMEM accumulators (the
// epilogue of tile i overlaps the MMAs of tile i+1), 4 epilogue warps.
// kBN = 256: one 256-column accumulator (N = 256 is the full-width single-SM
// MMA), 8 epilogue warps that copy it to registers and release TMEM before
// they convert and store, so the next tile's MMAs start almost at once.
//
// kARows = 64 (tokens T <= 64, the decode shapes): only 64 A rows are loaded per
// stage (8 KiB instead of 16); the MMA still reads a 128-row A tile, whose last
// 64 rows (the next bytes of shared memory) only reach accumulator rows that
// are never stored.  The smaller stage fits 8 stages instead of 6, a third more
// weight bytes in flight per CTA.
//
// kKps = 2: a pipeline stage holds two consecutive k-blocks (eight MMAs) behind
// one full and one empty barrier, so the MMA thread waits and commits once
// per eight MMAs instead of once per four.  The tensor pipe only stays busy if
// the issuing thread queues MMAs faster than it drains them; a barrier wait
// between groups of four MMAs measured ~0.7-0.8 of the ideal issue rate even
// with operands resident, a wait per eight 1.0.  The shared memory holds the
// same k-blocks (kSlots), in half as many stages.
template <int kBN, int kARows = 128, bool kFused = false, int kKps = 1>
struct Cfg {
  static_assert(kKps == 1 || (kKps == 2 && !kFused), "two k-blocks per stage: unfused A only");
  static constexpr uint32_t kABytes = kARows * kBK;
  // k-block buffers (A and B tiles) and the stages that group them
  static constexpr int kSlots = kFused ? 6 : (kARows == 64) ? 8 : (kBN == 128) ? 6 : 4;
  static constexpr int kStages = kSlots / kKps;
  static constexpr int kAccBufs = (kBN == 128) ? 2 : 1;
  static constexpr int kEpiWarps = (kBN == 128) ? 4 : 8;
  static constexpr int kEpiWarp0 = 3;
  // fused A (kFused): four producer warps after the epilogue warps build the
  // A tile from the attention output (16 token rows each)
  static constexpr int kProdWarps = kFused ? 4 : 0;
  static constexpr int kProdWarp0 = kEpiWarp0 + kEpiWarps;
  static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps + kProdWarps);
  static constexpr uint32_t kBBytes = kBN * kBK;
  static constexpr int kSfSlots = kStages;   // one scale-factor slot per stage (a stage
                                             // holds at most one pack start, see the kernel)
  static constexpr uint32_t kSfbBytes = kBN * 4;
  static constexpr uint32_t kSfSlotBytes = kSfaBytes + kSfbBytes;
  static constexpr int kSfCol0 = kAccBufs * kBN;              // after the accumulators
  static constexpr int kSfColsPerSlot = 4 + kBN / 32;         // A: 4, B: kBN/32
  static_assert(kSfCol0 + kSfSlots * kSfColsPerSlot <= kTmemCols, "TMEM budget");
  // shared memory plan (operand tiles 1024-byte aligned for the 128B swizzle)
  static constexpr uint32_t a = 0;
  static constexpr uint32_t b = a + kSlots * kABytes;
  static constexpr uint32_t sf = b + kSlots * kBBytes;
  // fused A: a ring of kOStages bf16 slices of the attention output (kARows
  // token rows x 128 elements of one head, 256 B a row), loaded by TMA ahead
  // of the producer warps
  static constexpr int kOStages = kFused ? 3 : 0;
  static constexpr uint32_t kOBytes = kARows * 256;
  static constexpr uint32_t ostage = (sf + kSfSlots * kSfSlotBytes + 1023) / 1024 * 1024;
  // per epilogue warp, a 2 KiB staging buffer for its TMA stores (32 rows x 64 B)
  static constexpr uint32_t kEpiBufBytes = 2048;
  // fused A: each token row's cos || sin cache row (64 fp32), copied per tile
  static constexpr uint32_t kCsBytes = kFused ? kARows * 256 : 0;
  static constexpr uint32_t csrows = ostage + kOStages * kOBytes;
  static constexpr uint32_t epi = csrows + kCsBytes;
  static constexpr uint32_t bars = epi + kEpiWarps * kEpiBufBytes;
  // full/empty[kStages], tmem_full/empty[kAccBufs], drain, o_full/o_empty[kOStages]
  static constexpr uint32_t n_bars = 2 * kStages + 2 * kAccBufs + 1 + 2 * kOStages;
  static constexpr uint32_t misc = bars + n_bars * 8;  // tmem base, abort flag
  static constexpr uint32_t total = misc + 16;
  static constexpr uint32_t smem_bytes = total + 1024;  // + alignment slack
};

// Tile schedule.  kSplit = 1: a persistent CTA walks tiles blockIdx.x,
// blockIdx.x + gridDim.x, ... over all k-blocks.  kSplit > 1: a cluster of
// kSplit CTAs shares one output tile, CTA r of the cluster taking k-blocks
// [r, r+1) * k_blocks / kSplit.  Each role evaluates these where it uses them:
// values computed once above the role dispatch stay live through every role
// and cost the tensor pipe a few per cent (measured).
template <int kSplit>
__device__ __forceinline__ int split_rank() {
  return kSplit > 1 ? static_cast<int>(cluster_cta_rank()) : 0;
}
template <int kSplit>
__device__ __forceinline__ int first_tile() {
  return kSplit > 1 ? static_cast<int>(blockIdx.x) / kSplit : static_cast<int>(blockIdx.x);
}
template <int kSplit>
__device__ __forceinline__ int tile_stride(const Params& p) {
  return kSplit > 1 ? p.num_tiles : static_cast<int>(gridDim.x);
}
template <int kSplit>
__device__ __forceinline__ int kb_begin(const Params& p) {
  return kSplit > 1 ? split_rank<kSplit>() * (p.k_blocks / kSplit) : 0;
}
template <int kSplit>
__device__ __forceinline__ int kb_end(const Params& p) {
  return kSplit > 1 ? kb_begin<kSplit>(p) + p.k_blocks / kSplit : p.k_blocks;
}

// Stages of kKps k-blocks: stage s holds the A and B tiles of its k-blocks in
// buffers kKps s .. kKps s + kKps - 1.  A k-range starts at an even k-block
// (0, or a multiple of four for the split-K halves), so a two-k-block stage
// never straddles a pack of four: only a stage's first k-block can start a
// pack.  The last stage of an odd k-range holds one k-block.
template <int kBN, int kEpi, int kSplit, bool kBf16, int kARows, bool kFused, int kKps>
__global__ void __launch_bounds__(Cfg<kBN, kARows, kFused, kKps>::kThreads, 1)
    block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                             const __grid_constant__ CUtensorMap tm_b,
                             const __grid_constant__ CUtensorMap tm_out, const Params p) {
  using C = Cfg<kBN, kARows, kFused, kKps>;
  static_assert(!kFused || (!kBf16 && kARows == 64 && kBN == 128), "fused A: decode tiles");
  static_assert(kSplit <= 2, "the split-K reduction has one partial buffer per warp slice");
  constexpr uint32_t kABytes = C::kABytes;
  constexpr int kStages = C::kStages;
  constexpr int kAccBufs = C::kAccBufs;
  constexpr uint32_t kBBytes = C::kBBytes;
  // elements of K per k-block: 128 e4m3 or 64 bf16 (128 bytes, one swizzle row)
  constexpr int kBKe = kBf16 ? 64 : kBK;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128B-swizzled operand tiles
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bars);
  uint64_t* full = bars;
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint64_t* tmem_empty = tmem_full + kAccBufs;
  uint64_t* drain = tmem_empty + kAccBufs;
  uint64_t* o_full = drain + 1;               // fused A: the attention-output ring
  uint64_t* o_empty = o_full + C::kOStages;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + C::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();  // a following GEMM may start its prologue now


  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // the producer's expect_tx, the scale-factor warp (FP8), the A producers (fused)
      mbar_init(&full[s], kBf16 ? 1 : 2 + C::kProdWarps);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kAccBufs; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], C::kEpiWarps);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < C::kOStages; ++i) {
      mbar_init(&o_full[i], 1);               // the TMA thread's expect_tx
      mbar_init(&o_empty[i], C::kProdWarps);  // every producer warp has read it
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if constexpr (!kFused) tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // bit s: stage s loaded / parity of its phase
      int oj = 0;                              // fused A: the o ring
      uint32_t ophase = 0, o_issued = 0, o_issued_parity = 0;
      bool ok = true;
      // Before the previous kernel of the stream has finished (programmatic
      // launch) only the weights may be read: the first stages of the first
      // tile get their B tile now and their A tile after griddep_wait().
      // bytes that land on a stage's full barrier for n k-blocks (fused A:
      // the producer warps write A; only B travels by TMA)
      auto stage_tx = [](int n) {
        return static_cast<uint32_t>(n) * (kFused ? kBBytes : kABytes + kBBytes);
      };
      int early = 0;   // stages
      if (first_tile<kSplit>() < p.num_tiles) {
        int g, n_blk, m_blk;
        tile_coords(p, first_tile<kSplit>(), g, n_blk, m_blk);
        const int brow = g * p.N + n_blk * kBN;
        const int kb0 = kb_begin<kSplit>(p), kb1 = kb_end<kSplit>(p);
        const int nst = (kb1 - kb0 + kKps - 1) / kKps;
        early = nst < kStages ? nst : kStages;
        for (int i = 0; i < early; ++i) {
          const int kbs = kb0 + i * kKps;
          const int n = (kKps == 1 || kb1 - kbs >= kKps) ? kKps : kb1 - kbs;
          mbar_arrive_expect_tx(&full[i], stage_tx(n));
          for (int j = 0; j < n; ++j)
            tma_load_2d(smem + C::b + (i * kKps + j) * kBBytes, &tm_b, &full[i],
                        (kbs + j) * kBKe, brow);
        }
        // The rest of the first tile's weights go to L2 while the previous
        // kernel still runs, so that the weight-bound small-T shapes stream
        // them from L2 once their activations are ready.
        if (p.prefetch_l2)
          for (int kb = kb0 + early * kKps; kb < kb1; ++kb)
            tma_prefetch_l2_2d(&tm_b, kb * kBKe, brow);
      }
      griddep_wait();
      for (int tile = first_tile<kSplit>(); tile < p.num_tiles && ok;
           tile += tile_stride<kSplit>(p)) {
        int g, n_blk, m_blk;
        tile_coords(p, tile, g, n_blk, m_blk);
        [[maybe_unused]] const int m0 = m_blk * kBM;
        const int brow = g * p.N + n_blk * kBN;
        for (int kbs = kb_begin<kSplit>(p); kbs < kb_end<kSplit>(p); kbs += kKps) {
          const int n = (kKps == 1 || kb_end<kSplit>(p) - kbs >= kKps) ? kKps
                                                                       : kb_end<kSplit>(p) - kbs;
          if constexpr (kFused) {
            const int kb = kbs;   // one k-block per stage
            // this k-block's slice of o: rows m0.., head g*hpg + kb/4, elements
            // (kb % 4)*128 .. +127 (rows past T zero-filled)
            if (!mbar_wait(&o_empty[oj], ophase ^ 1u, abort_flag, p.status)) { ok = false; break; }
            mbar_arrive_expect_tx(&o_full[oj], C::kOBytes);
            tma_load_2d(smem + C::ostage + oj * C::kOBytes, &tm_a, &o_full[oj],
                        (g * p.hpg + (kb >> 2)) * 512 + (kb & 3) * 128, m0);
            o_issued |= 1u << oj;
            o_issued_parity = (o_issued_parity & ~(1u << oj)) | (ophase << oj);
            if (++oj == C::kOStages) { oj = 0; ophase ^= 1u; }
          }
          if (early > 0) {  // B already in flight for this stage
            if constexpr (!kFused)
              for (int j = 0; j < n; ++j)
                tma_load_3d(smem + C::a + (stage * kKps + j) * kABytes, &tm_a, &full[stage],
                            (kbs + j) * kBKe, m0, g);
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
            --early;
            continue;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], stage_tx(n));
          for (int j = 0; j < n; ++j) {
            if constexpr (!kFused)
              tma_load_3d(smem + C::a + (stage * kKps + j) * kABytes, &tm_a, &full[stage],
                          (kbs + j) * kBKe, m0, g);
            tma_load_2d(smem + C::b + (stage * kKps + j) * kBBytes, &tm_b, &full[stage],
                        (kbs + j) * kBKe, brow);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // drain: let every copy issued here land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) mbar_wait_drain(&full[s], (issued_parity >> s) & 1u);
        for (int s = 0; s < C::kOStages; ++s)
          if (o_issued & (1u << s)) mbar_wait_drain(&o_full[s], (o_issued_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issue
      const uint64_t adesc0 = smem_desc(smem_addr(smem + C::a), 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_addr(smem + C::b), 16, 1024, 2);
      const uint64_t sfdesc0 = smem_desc(smem_addr(smem + C::sf), 0, 128, 0);
      // The scale-factor id (the k-block within its pack of four) selects the
      // byte of the packed scale words: fields [4,6) (B) and [29,31) (A) of the
      // instruction descriptor, set arithmetically (an indexed array of four
      // descriptors would live in local memory).
      const uint32_t idesc0 = kBf16 ? bf16_idesc(kBM, kBN) : mxf8_idesc(kBM, kBN, 0, 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // A pack's scale words serve its four k-blocks (the scale-factor id picks
      // the byte), so they are copied to TMEM once per pack, into region
      // (packs so far) mod kStages.  A region is rewritten kStages packs later,
      // by which time the full-barrier wait of that stage proves every MMA at
      // least kStages stages back complete, the old pack's included.  (The
      // fused A role writes one byte per stage; it copies every stage.)
      int sf_region = kStages - 1;
      for (int tile = first_tile<kSplit>(); tile < p.num_tiles && ok;
           tile += tile_stride<kSplit>(p)) {
        if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        const int kb0 = kb_begin<kSplit>(p);
        for (int kbs = kb0; kbs < kb_end<kSplit>(p); kbs += kKps) {
          const int n = (kKps == 1 || kb_end<kSplit>(p) - kbs >= kKps) ? kKps
                                                                       : kb_end<kSplit>(p) - kbs;
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          // the stage's scale factors arrived with its operands (same barrier)
          const bool pack_start = kbs == kb0 || (kbs & 3) == 0;
          if (pack_start) sf_region = (sf_region + 1 == kStages) ? 0 : sf_region + 1;
          const uint32_t sf_col = tmem_base + static_cast<uint32_t>(
              C::kSfCol0 + (kFused ? stage : sf_region) * C::kSfColsPerSlot);
          if (!kBf16 && (kFused || pack_start)) {
            const uint64_t sd = sfdesc0 + ((stage * C::kSfSlotBytes) >> 4);
            tmem_cp_32x128b_x4(sf_col, sd);                     // A: the slot's first 512 B
#pragma unroll
            for (int r = 0; r < kBN / 128; ++r)                 // B: 512 B per 128 rows
              tmem_cp_32x128b_x4(sf_col + 4 + 4 * r, sd + ((kSfaBytes + 512u * r) >> 4));
          }
#pragma unroll
          for (int j = 0; j < kKps; ++j) {
            if (j < n) {
              const int kb = kbs + j;
              const uint64_t ad = adesc0 + (((stage * kKps + j) * kABytes) >> 4);
              const uint64_t bd = bdesc0 + (((stage * kKps + j) * kBBytes) >> 4);
              const uint32_t sfid = kBf16 ? 0u : static_cast<uint32_t>(kb & 3);
              const uint32_t id = idesc0 | (sfid << 4) | (sfid << 29);
              // four MMAs per k-block: K = 32 e4m3 or K = 16 bf16, 32 bytes each
              // (+32 bytes along K = +2 in the descriptor's address field)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if constexpr (kBf16)
                  mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, id, ((kb - kb0) | k) != 0 ? 1u : 0u);
                else
                  mma_mxf8(d_tmem, ad + 2 * k, bd + 2 * k, id, sf_col, sf_col + 4,
                           ((kb - kb0) | k) != 0 ? 1u : 0u);
              }
            }
          }
          mma_commit(&empty[stage]);   // frees the stage's operands and scale-factor slot
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&tmem_full[acc]);
        if (++acc == kAccBufs) { acc = 0; acc_phase ^= 1u; }
      }
      if (*abort_flag) {
        // let every MMA / copy this thread issued finish before TMEM is freed
        mma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else if (warp == 2 && !kBf16) {
    // ------------------------------------------------------ scale factors
    constexpr int kRb = kBN / 128;   // 128-row weight-scale blocks per tile
    const int packs = p.packs;
    uint32_t wnext[kRb][4];
#pragma unroll
    for (int r = 0; r < kRb; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) wnext[r][i] = 0u;
    if (first_tile<kSplit>() < p.num_tiles) {
      int g, nb, mb;
      tile_coords(p, first_tile<kSplit>(), g, nb, mb);
      const int rb = (g * p.N + nb * kBN) / 128;
#pragma unroll
      for (int r = 0; r < kRb; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (lane + 32 * i < packs) wnext[r][i] = b_scale_word(p, rb + r, lane + 32 * i);
    }
    griddep_wait();  // the A scale words are written by the previous kernel
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = first_tile<kSplit>(); tile < p.num_tiles && ok;
         tile += tile_stride<kSplit>(p)) {
      int g, n_blk, m_blk;
      tile_coords(p, tile, g, n_blk, m_blk);
      uint32_t wcur[kRb][4];
#pragma unroll
      for (int r = 0; r < kRb; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) wcur[r][i] = wnext[r][i];
      const int next = tile + tile_stride<kSplit>(p);
      if (next < p.num_tiles) {
        int g2, nb2, mb2;
        tile_coords(p, next, g2, nb2, mb2);
        const int rb2 = (g2 * p.N + nb2 * kBN) / 128;
#pragma unroll
        for (int r = 0; r < kRb; ++r)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            wnext[r][i] = (lane + 32 * i < packs) ? b_scale_word(p, rb2 + r, lane + 32 * i) : 0u;
      }
      const int64_t m0 = static_cast<int64_t>(m_blk) * kBM;
      // the 128 A scale words of pack j: lane r takes rows r, r+32, r+64, r+96
      auto load_pack = [&](int j, uint32_t (&v)[4]) {
        const int32_t* src = p.a_scale + (static_cast<int64_t>(g) * packs + j) * p.t_al + m0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t t = m0 + 32 * c + lane;
          v[c] = (j < packs && t < p.T) ? static_cast<uint32_t>(__ldg(src + 32 * c + lane)) : 0u;
        }
      };
      const int kb0 = kb_begin<kSplit>(p);
      uint32_t vcur[4] = {0u, 0u, 0u, 0u}, vnext[4] = {0u, 0u, 0u, 0u};
      if constexpr (!kFused) load_pack(kb0 / 4, vnext);   // fused A: the producers write SFA
      uint32_t bword[kRb];
      for (int kbs = kb0; kbs < kb_end<kSplit>(p); kbs += kKps) {
        const bool pack_start = kbs == kb0 || (kbs & 3) == 0;
        if (pack_start) {   // a new pack: its words, and the next pack's load
          const int j = kbs / 4;
          if constexpr (!kFused) {
#pragma unroll
            for (int c = 0; c < 4; ++c) vcur[c] = vnext[c];
            load_pack(j + 1, vnext);
          }
#pragma unroll
          for (int r = 0; r < kRb; ++r) {
            const uint32_t src_w = (j < 32) ? wcur[r][0] : (j < 64) ? wcur[r][1]
                                 : (j < 96) ? wcur[r][2] : wcur[r][3];
            bword[r] = __shfl_sync(0xFFFFFFFFu, src_w, j & 31);
          }
        }
        // fused A: the producer warps need the issue slots, so this warp sleeps
        const bool got = kFused
            ? mbar_wait_warp_lazy(&empty[stage], phase ^ 1u, abort_flag, p.status, 64)
            : mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag, p.status);
        if (!got) { ok = false; break; }
        // The MMA thread copies a slot to TMEM only at the first k-block of a
        // pack (fused A: every k-block, whose A scale byte the producers write),
        // so only those slots are written; for the others this warp only
        // arrives once the stage is free.
        if (kFused || pack_start) {
          uint4* dst = reinterpret_cast<uint4*>(smem + C::sf + stage * C::kSfSlotBytes);
          if constexpr (!kFused) dst[lane] = make_uint4(vcur[0], vcur[1], vcur[2], vcur[3]);
#pragma unroll
          for (int r = 0; r < kRb; ++r)
            dst[32 + 32 * r + lane] = make_uint4(bword[r], bword[r], bword[r], bword[r]);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (kFused && warp >= C::kProdWarp0) {
    // ---------------------------------------------- fused A producer (T <= 64)
    // Builds each stage's A tile from the attention output: the inverse
    // rotation, the per-128 block scale and the e4m3 cast of the quantiser
    // (the same helpers, so the same codes and scales bit for bit), written in
    // the 128-byte-swizzled layout the MMA reads (16-byte unit u of row r at
    // u ^ (r & 7)), and each row's scale byte, as byte kb % 4 of its word in
    // the stage's scale-factor slot.  The k-block's bf16 slice arrives by TMA
    // in the o ring; a half-warp owns one token row (lane l16 holds its
    // elements 8 l16 .. 8 l16 + 7, 16 contiguous bytes of the row's 256);
    // warp pw owns rows 16 pw .. 16 pw + 15, two per step.  Each row's
    // cos || sin cache row is copied into shared memory once per tile and
    // read at the rope block of each head (held in registers for all rows,
    // the values spilled and the warp took ~3000 cycles per k-block).
    constexpr int kSteps = kARows / (2 * (C::kProdWarps > 0 ? C::kProdWarps : 1));
    const int pw = warp - C::kProdWarp0;
    const int half = lane >> 4;
    const int l16 = lane & 15;
    const bool rope_lane = l16 >= 8;     // block 3: head offsets 448 .. 511
    const int quad = l16 - 8;            // rope pairs 4 quad .. 4 quad + 3
    int stage = 0, oj = 0;
    uint32_t phase = 0, ophase = 0;
    bool ok = true;
    for (int tile = first_tile<kSplit>(); tile < p.num_tiles && ok;
         tile += tile_stride<kSplit>(p)) {
      int g, n_blk, m_blk;
      tile_coords(p, tile, g, n_blk, m_blk);
      const int64_t m0 = static_cast<int64_t>(m_blk) * kBM;
      // each row's position; one outside [0, max_pos) is recorded and leaves
      // the row unrotated, as in the quantiser.  Lane l16 copies float4 l16
      // of the row's cache row (cos: 0..7, sin: 8..15).
      float4* cs_rows = reinterpret_cast<float4*>(smem + C::csrows);   // [kARows][16]
      uint32_t rot_mask = 0;
      __syncwarp();   // the previous tile's reads of this warp's rows are done
#pragma unroll
      for (int st = 0; st < kSteps; ++st) {
        const int r = 16 * pw + 2 * st + half;
        const int64_t t = m0 + r;
        float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < p.T) {
          const int64_t pos = __ldg(p.positions + t);
          if (pos >= 0 && pos < p.max_pos) {
            rot_mask |= 1u << st;
            cv = __ldg(reinterpret_cast<const float4*>(p.cache + pos * 64) + l16);
          } else if (l16 == 0) {
            record_status(p.status, DSV4_ERR_RANGE);
          }
        }
        cs_rows[r * 16 + l16] = cv;
      }
      __syncwarp();
      for (int kb = kb_begin<kSplit>(p); kb < kb_end<kSplit>(p); ++kb) {
        const int qb = kb & 3;
        if (!mbar_wait_warp(&o_full[oj], ophase, abort_flag, p.status)) { ok = false; break; }
        const uint4* slice = reinterpret_cast<const uint4*>(smem + C::ostage + oj * C::kOBytes);
        uint4 v[kSteps];
#pragma unroll
        for (int st = 0; st < kSteps; ++st) v[st] = slice[(16 * pw + 2 * st + half) * 16 + l16];
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_empty[oj]);   // the slice is in registers
        if (++oj == C::kOStages) { oj = 0; ophase ^= 1u; }
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
        uint8_t* a_st = smem + C::a + stage * kABytes;
        uint32_t* sfa = reinterpret_cast<uint32_t*>(smem + C::sf + stage * C::kSfSlotBytes);
        // The eight rows are independent: their maxima are reduced together
        // (each shuffle level for all rows before the next), so the shuffle
        // latencies overlap; the values are unpacked (and rotated) again for
        // the cast instead of being held.
        auto values = [&](int st, float (&f)[8]) {
          unpack8(v[st], f);
          if (qb == 3 && rope_lane && ((rot_mask >> st) & 1u)) {
            const int r = 16 * pw + 2 * st + half;
            const float4 c = cs_rows[r * 16 + quad];
            const float4 sn = cs_rows[r * 16 + 8 + quad];
            inv_rotate(f[0], f[1], c.x, sn.x);
            inv_rotate(f[2], f[3], c.y, sn.y);
            inv_rotate(f[4], f[5], c.z, sn.z);
            inv_rotate(f[6], f[7], c.w, sn.w);
          }
        };
        float m[kSteps];
#pragma unroll
        for (int st = 0; st < kSteps; ++st) {
          float f[8];
          values(st, f);
          m[st] = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) m[st] = fmaxf(m[st], fabsf(f[j]));
        }
#pragma unroll
        for (int mask = 8; mask >= 1; mask >>= 1)
#pragma unroll
          for (int st = 0; st < kSteps; ++st)
            m[st] = fmaxf(m[st], __shfl_xor_sync(0xFFFFFFFFu, m[st], mask));
#pragma unroll
        for (int st = 0; st < kSteps; ++st) {
          float f[8];
          values(st, f);
          const int e = ue8m0_exponent(m[st]);
          const uint2 q = quant8(f, exp2_neg(e));
          const int r = 16 * pw + 2 * st + half;
          *reinterpret_cast<uint2*>(a_st + r * 128 + ((((l16 >> 1) ^ (r & 7)) << 4) |
                                                      ((l16 & 1) << 3))) = q;
          // scale word of row r: lane r % 32, column r / 32 of the slot's A part
          if (l16 == 0) sfa[(r & 31) * 4 + (r >> 5)] = static_cast<uint32_t>(e + 127) << (8 * qb);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int epi = warp - C::kEpiWarp0;  // 0 .. kEpiWarps-1
    const int quarter = warp & 3;         // TMEM lanes this warp may access
    const int col_half = epi >> 2;        // which 128 columns of the tile
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool synced = false;  // split-K: this warp took part in the two cluster barriers
    for (int tile = first_tile<kSplit>(); tile < p.num_tiles;
         tile += tile_stride<kSplit>(p)) {
      int g, n_blk, m_blk;
      tile_coords(p, tile, g, n_blk, m_blk);
      // fused A: the accumulator wait spans the mainloop; sleep instead of spinning
      const bool got = kFused
          ? mbar_wait_warp_lazy(&tmem_full[acc], acc_phase, abort_flag, p.status, 128)
          : mbar_wait_warp(&tmem_full[acc], acc_phase, abort_flag, p.status);
      if (!got) break;
      tc_fence_after();
      const int64_t t = static_cast<int64_t>(m_blk) * kBM + row;
      const bool live = t < p.T;
      const int64_t col0 = static_cast<int64_t>(g) * p.N + static_cast<int64_t>(n_blk) * kBN +
                           128 * col_half;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * kBN + 128 * col_half);
      // the whole 128-column slice to registers, then hand the accumulator back
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32cols(taddr + 32u * c, r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[acc]);
      if constexpr (kSplit > 1) {
        // Split-K: the other CTAs of the cluster add their partial tiles into
        // this one.  Every pipeline of the cluster has drained by the first
        // barrier, so the leader's A stage buffers are free; each warp slice
        // (32 rows x 128 fp32) has its own 16 KiB there, laid out [col/4][lane].
        cluster_sync();
        const uint32_t part = smem_addr(smem + C::a) + static_cast<uint32_t>(epi) * 16384u;
        // a warp whose 32 rows all lie past the last token has nothing to add
        // (those rows are never stored): it only meets the two barriers
        const bool rows_live = static_cast<int64_t>(m_blk) * kBM + quarter * 32 < p.T;
        if (split_rank<kSplit>() != 0 && rows_live) {
          const uint32_t dst = map_to_cta(part, 0);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int v = 0; v < 8; ++v)
              st_cluster_v4(dst + static_cast<uint32_t>(((c * 8 + v) * 32 + lane) * 16),
                            r[c][4 * v], r[c][4 * v + 1], r[c][4 * v + 2], r[c][4 * v + 3]);
        }
        cluster_sync();
        synced = true;
        if (split_rank<kSplit>() == 0 && rows_live) {
          for (int peer = 1; peer < kSplit; ++peer) {
            const float4* src = reinterpret_cast<const float4*>(smem + C::a + epi * 16384);
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const float4 q = src[(c * 8 + v) * 32 + lane];
                r[c][4 * v] = __float_as_uint(__uint_as_float(r[c][4 * v]) + q.x);
                r[c][4 * v + 1] = __float_as_uint(__uint_as_float(r[c][4 * v + 1]) + q.y);
                r[c][4 * v + 2] = __float_as_uint(__uint_as_float(r[c][4 * v + 2]) + q.z);
                r[c][4 * v + 3] = __float_as_uint(__uint_as_float(r[c][4 * v + 3]) + q.w);
              }
          }
        }
      }
      if (split_rank<kSplit>() == 0) {
      // Stores go through this warp's staging buffer: each lane writes its row's
      // 64-byte chunk with the 64-byte TMA swizzle (16-byte unit q of row r at
      // q ^ ((r >> 1) & 3): conflict-free), then one lane stores the 32-row box
      // with TMA, which also clips rows beyond T.
      uint8_t* buf = smem + C::epi + epi * C::kEpiBufBytes;
      const int32_t box_y = static_cast<int32_t>(static_cast<int64_t>(m_blk) * kBM + quarter * 32);
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
        // eight chunks of 16 columns (64 bytes of fp32 per row), the
        // accumulators unchanged
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int b = 16 * (c & 1) + 4 * q;
            v[q] = make_uint4(r[c >> 1][b], r[c >> 1][b + 1], r[c >> 1][b + 2], r[c >> 1][b + 3]);
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
              const int b = 16 * (q & 1) + 4 * i;
              w[i] = static_cast<uint32_t>(e4m3x2(__uint_as_float(r[c][b]) * inv,
                                                  __uint_as_float(r[c][b + 1]) * inv)) |
                     (static_cast<uint32_t>(e4m3x2(__uint_as_float(r[c][b + 2]) * inv,
                                                   __uint_as_float(r[c][b + 3]) * inv))
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
      }  // split rank 0
      if (++acc == kAccBufs) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();   // every store complete before the CTA leaves
    __syncwarp();
    if (kSplit > 1 && !synced) {       // aborted before the reduction: still meet the cluster
      cluster_sync();
      cluster_sync();
    }
  }
  if constexpr (kSplit > 1) {
    // every thread of the cluster meets both barriers of the reduction:
    // the producer, MMA and scale-factor warps (and the fused A producers) here
    if (warp < C::kEpiWarp0 || (kFused && warp >= C::kProdWarp0)) {
      __syncwarp();                    // lane 0 of warps 0 and 1 finished its loop
      cluster_sync();
      cluster_sync();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int kBN, int kEpi, int kSplit, bool kBf16, int kARows, bool kFused = false,
          int kKps = 1>
int launch_impl(const GemmProblem& q, cudaStream_t stream, const DeviceInfo& dev) {
  // q.after_own_kernel: the previous kernel on the stream does not write the
  // weights (inside dsv4_o_proj it is one of this library's), so the launch
  // may overlap it: this kernel reads only weights before griddep_wait().
  using C = Cfg<kBN, kARows, kFused, kKps>;
  static std::atomic<int> configured_for[kMaxDevices];
  if (dev.device < 0 || dev.device >= kMaxDevices) return DSV4_ERR_UNSUPPORTED;
  const int configured = lazy_per_device(configured_for, dev.device, [] {
    return cudaFuncSetAttribute(block_scaled_gemm_kernel<kBN, kEpi, kSplit, kBf16, kARows, kFused,
                                                         kKps>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::smem_bytes)) == cudaSuccess ? 1 : 0;
  });
  if (!configured) return DSV4_ERR_CUDA;
  const int64_t T = q.T;
  const int64_t t_al = (T + 3) / 4 * 4;
  const int packs = (q.K / 128 + 3) / 4;

  // operands: 128-byte rows of K (128 e4m3 or 64 bf16 elements) per k-block
  const int esz = kBf16 ? 2 : 1;
  const int kbe = kBK / esz;
  const CUtensorMapDataType dt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap tm_a, tm_b;
  if (kFused) {
    // fused A: tm_a maps the attention output o as [T][H*512] bf16; a box is
    // kARows token rows x 128 elements (one head's k-block), rows past T
    // zero-filled
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(q.heads) * 512, static_cast<cuuint64_t>(T)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(q.heads) * 512 * 2};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(kARows)};
    if (!encode(&tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q.o, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE))
      return DSV4_ERR_CUDA;
  } else {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(q.K), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(q.G)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(q.K) * esz,
                             static_cast<cuuint64_t>(T * q.K) * esz};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kbe), static_cast<cuuint32_t>(kARows), 1};
    if (!encode(&tm_a, dt, 3, q.a, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return DSV4_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(q.K),
                          static_cast<cuuint64_t>(static_cast<int64_t>(q.G) * q.N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(q.K) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kbe), kBN};
    if (!encode(&tm_b, dt, 2, q.b, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return DSV4_ERR_CUDA;
  }
  CUtensorMap tm_out;
  {
    // rows of G*N elements; a box is 32 rows x 64 bytes (64 e4m3 codes, 32
    // bf16 or 16 fp32 values)
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
  Params p;
  p.T = T;
  p.G = q.G;
  p.N = q.N;
  p.K = q.K;
  p.m_tiles = static_cast<int>((T + kBM - 1) / kBM);
  p.n_tiles = q.N / kBN;
  p.num_tiles = p.m_tiles * p.n_tiles * q.G;
  p.k_blocks = q.K / kbe;
  p.packs = packs;
  p.t_al = t_al;
  p.a_scale = q.a_scale;
  p.b_scale = q.b_scale;
  p.b_scale_ld = q.K / 128;
  p.out = static_cast<__nv_bfloat16*>(q.out_bf16);
  p.q_out = q.q_out;
  p.q_scale = q.q_scale;
  p.status = dev.status;
  p.o = q.o;
  p.positions = q.positions;
  p.cache = q.cache;
  p.max_pos = q.max_pos;
  p.H = q.heads;
  p.hpg = q.heads_per_group;
  p.raster_m = (q.G == 1 && p.m_tiles > kRasterM) ? kRasterM : 0;
  p.prefetch_l2 = q.after_own_kernel ? 1 : 0;

  // persistent: one CTA per SM; split-K: one cluster of kSplit CTAs per tile
  const int grid = kSplit == 1 ? (p.num_tiles < dev.num_sms ? p.num_tiles : dev.num_sms)
                               : p.num_tiles * kSplit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (kSplit > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = kSplit;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (q.after_own_kernel) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg,
                         block_scaled_gemm_kernel<kBN, kEpi, kSplit, kBf16, kARows, kFused, kKps>,
                         tm_a, tm_b, tm_out, p) != cudaSuccess)
    return DSV4_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

// The FP8 tile paths for one epilogue: two k-blocks per stage (their k-ranges
// start at 0 or, split over K, at a multiple of four k-blocks).
template <int kEpi>
int launch_fp8(const GemmProblem& q, bool wide, bool small_m, bool split, cudaStream_t stream,
               const DeviceInfo& dev) {
  if (wide) return launch_impl<256, kEpi, 1, false, 128, false, 1>(q, stream, dev);
  if (small_m) {
    if (split) return launch_impl<128, kEpi, 2, false, 64, false, 2>(q, stream, dev);
    return launch_impl<128, kEpi, 1, false, 64, false, 2>(q, stream, dev);
  }
  if (split) return launch_impl<128, kEpi, 2, false, 128, false, 2>(q, stream, dev);
  return launch_impl<128, kEpi, 1, false, 128, false, 2>(q, stream, dev);
}

}  // namespace

int launch_block_scaled_gemm(const GemmProblem& q, cudaStream_t stream, const DeviceInfo& dev) {
  if (q.K / 128 > 4 * 32 * 4) return DSV4_ERR_UNSUPPORTED;  // weight-scale words held per lane
  if (q.fused_a) {
    // decode sizes only: one 64-row m-tile, 128-wide tiles, split over K when
    // both halves hold whole scale packs and the split still fits the GPU
    if (q.bf16 || q.T > 64 || q.N % 128 != 0 || q.K != q.heads_per_group * 512 ||
        q.epilogue == kEpiF32)
      return DSV4_ERR_UNSUPPORTED;
    const int64_t tiles = static_cast<int64_t>(q.N / 128) * q.G;
    const bool split = (q.K / 128) % 8 == 0 && 2 * tiles <= dev.num_sms;
    const bool quant = q.epilogue == kEpiQuant;
    if (split) {
      if (quant) return launch_impl<128, kEpiQuant, 2, false, 64, true>(q, stream, dev);
      return launch_impl<128, kEpiBf16, 2, false, 64, true>(q, stream, dev);
    }
    if (quant) return launch_impl<128, kEpiQuant, 1, false, 64, true>(q, stream, dev);
    return launch_impl<128, kEpiBf16, 1, false, 64, true>(q, stream, dev);
  }
  // Large shapes (FP8, and bf16 with the bf16 epilogue): 256 x 256 tiles on CTA
  // pairs (two thirds of the shared-memory operand bytes per SM and k-block,
  // three two-k-block stages)
  if (pair_gemm_eligible(q, dev)) return launch_pair_gemm(q, stream, dev);
  // 256-wide tiles when they divide N and still give every SM a tile;
  // otherwise 128-wide tiles (twice the CTAs, for the small decode shapes)
  const int64_t m_tiles = (q.T + kBM - 1) / kBM;
  const bool wide = q.N % 256 == 0 && m_tiles * (q.N / 256) * q.G >= dev.num_sms;
  // Too few 128-wide tiles to fill the GPU (decode): split K over a 2-CTA
  // cluster when both halves hold whole k-blocks (and, for FP8, whole scale
  // packs: k_blocks % 8 == 0).
  const int64_t tiles = m_tiles * (q.N / 128) * q.G;
  const int kbs = q.bf16 ? q.K / 64 : q.K / 128;
  const bool split = !wide && kbs % (q.bf16 ? 2 : 8) == 0 && 2 * tiles <= dev.num_sms;
  // at most 64 tokens: one m-tile with a 64-row A box (see Cfg)
  const bool small_m = !wide && q.T <= 64;
  if (q.bf16) {
    if (q.epilogue != kEpiBf16) return DSV4_ERR_UNSUPPORTED;
    if (wide) return launch_impl<256, kEpiBf16, 1, true, 128>(q, stream, dev);
    if (small_m) {
      if (split) return launch_impl<128, kEpiBf16, 2, true, 64>(q, stream, dev);
      return launch_impl<128, kEpiBf16, 1, true, 64>(q, stream, dev);
    }
    if (split) return launch_impl<128, kEpiBf16, 2, true, 128>(q, stream, dev);
    return launch_impl<128, kEpiBf16, 1, true, 128>(q, stream, dev);
  }
  switch (q.epilogue) {
    case kEpiQuant: return launch_fp8<kEpiQuant>(q, wide, small_m, split, stream, dev);
    case kEpiF32: return launch_fp8<kEpiF32>(q, wide, small_m, split, stream, dev);
    default: return launch_fp8<kEpiBf16>(q, wide, small_m, split, stream, dev);
  }
}

}  // namespace dsv4
