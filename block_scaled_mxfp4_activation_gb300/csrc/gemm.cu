// Block-scaled MXFP4 GEMM on the 5th-generation tensor cores (tcgen05,
// kind::mxf4, UE8M0 scales), with the activation quantized in the kernel
// (fused entry) or read pre-quantized.
//
// The pages' kernels (`kernel_fused_mxfp4_gemm` of submission 748756,
// `_tiled_gemm_engine` of submission 754569, the fused split-K kernels of
// submission 755056) quantize a bf16 A tile in registers, load packed FP4 B
// and its scales, and call `tl.dot_scaled` per K tile, with split-K partials
// reduced by a second kernel.  Here, per CTA:
//
//   - the output tile is C^T[128 weight rows, block_m activation rows]: the
//     weights are the MMA's A operand (M = 128) and the activations its B
//     operand (N = block_m), so a handful of tokens still fills the MMA;
//   - warp 0 issues every load of the CTA at once with TMA: per 256-wide K
//     tile, the 128 x 128-byte box of weight codes (128-byte swizzle), the
//     tile's 1 KB of pre-arranged weight scales (bulk copy) and, except on
//     the direct path, the activation tile -- bf16 for the fused entry, codes
//     straight into the MMA operand's swizzled layout for the unfused one
//     (fused, with weights loaded ahead of the grid wait: the first stages'
//     weights are issued by thread 0 as soon as it has initialised their
//     barriers, before the rest of the set-up);
//   - warps 2.. quantize the activation (fused: at block_m 16 and 32 loaded
//     straight from global memory into registers, else from the bf16 tile
//     staged in shared memory) or place the pre-quantized scales, writing
//     codes in the operand's swizzled layout and scales in the tensor-memory
//     scale-chunk layout;
//   - one lane of warp 1 moves both scale sets to tensor memory (tcgen05.cp)
//     and issues four K = 64 block-scaled MMAs per stage into an fp32
//     accumulator in tensor memory;
//   - without a K split, the accumulator leaves as bf16 through a tile in
//     shared memory and one TMA tensor store;
//   - K splits of one output tile form a thread-block cluster: each CTA
//     pushes its fp32 partial blocks into their owners' shared memory with
//     st.async, counted on the owner's barrier, and every owner sums its
//     blocks over the splits in a fixed order (deterministic, no global
//     workspace, no second kernel), then stores 8 bytes per thread.
//
// Back-to-back calls overlap through programmatic dependent launch: the next
// call's CTAs set up and load their weights into shared memory while this one
// runs (at most one call ahead).
#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "tile.cuh"

namespace mxfp4 {

template <int BM, bool kFused>
struct TileCfg {
  static constexpr int kRowChunks = BM > 128 ? 2 : 1;             // 128-row scale chunks of A
  static constexpr int kBTileBytes = kTileN * kTileKBytes;         // 16 KB of weight codes
  static constexpr int kATileBytes = BM * kTileKBytes;             // activation codes
  static constexpr int kSfaStageBytes = 2 * kRowChunks * kSfChunkBytes;
  static constexpr int kAWarps = 8;                                // producer / epilogue warps
  static constexpr int kAThreads = kAWarps * 32;
  static constexpr int kThreads = 64 + kAThreads;
  static constexpr int kSfCols = 8 + 8 * kRowChunks;               // TMEM scale columns per stage
  static_assert(BM == 16 || BM == 32 || BM == 64 || BM == 128 || BM == 256, "block_m must be 16, 32, 64, 128 or 256");
};

// The accumulator tile (128 weight rows x BM activation rows) is reduced over
// K splits in blocks of 32 weight rows (one TMEM lane quarter) x 16 activation
// rows (one tcgen05.ld): 2 KB of fp32 each.
constexpr int kBlockBytes = 32 * 16 * 4;

// Quantizes one staged bf16 activation tile [BM rows][256] (512-byte rows) into
// the MMA operand's codes (128-byte rows, 128-byte swizzle) and the scale
// chunks, with the kAThreads producer threads: two lanes per 32-element block
// (16 bf16 each), unit u = tid + kAThreads * k is row u / 16, block (u / 2) % 8,
// half u % 2, so warp w covers rows 2w + 16k and 2w + 16k + 1.  kGuard: rows
// past m_valid are skipped (a whole warp's unit at once, so the pair shuffle
// stays convergent; their output columns are never stored).
template <int BM, int kThreads, int kRowChunks, bool kGuard>
__device__ __forceinline__ void quantize_tile(const uint8_t* abf, uint8_t* a_tile, uint8_t* sfa, int tid, int m_valid) {
  constexpr int kUnits = BM * 16 / kThreads;
  const int lane = tid & 31, pw = tid >> 5;
  const int rot = (lane >> 2) & 1;  // which half of its 32 bytes a lane loads first: no bank conflicts
  const int half = lane & 1;        // which 16 elements of the block the lane owns
  // (batches of at most 4 units, 2 at block_m >= 128, to fit the register
  // budget of two CTAs per SM)
  constexpr int kBatch = kUnits < (BM < 128 ? 4 : 2) ? kUnits : (BM < 128 ? 4 : 2);
#pragma unroll(BM < 256 ? kUnits / kBatch : 1)
  for (int k0 = 0; k0 < kUnits; k0 += kBatch) {
    uint4 v[kBatch][2];  // all loads of a batch first, then the independent chains
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const uint8_t* src = abf + (tid + (k0 + e) * kThreads) * 32;
      if (!kGuard || 2 * pw + 16 * (k0 + e) < m_valid) {
        v[e][0] = *reinterpret_cast<const uint4*>(src + 16 * rot);  // 16 bytes rot, then 16 bytes rot ^ 1
        v[e][1] = *reinterpret_cast<const uint4*>(src + 16 * (rot ^ 1));
      }
    }
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      if (kGuard && 2 * pw + 16 * (k0 + e) >= m_valid) continue;  // warp-uniform
      const int u = tid + (k0 + e) * kThreads;
      const int m = u >> 4, b = (u >> 1) & 7;
      uint32_t amax = absmax16_bf16(v[e][0], v[e][1]);
      amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      const uint32_t byte = scale_byte_from_amax(amax);
      const uint16_t sbf = scale_bf16_from_byte(byte);
      uint32_t w0 = e2m1_pack8(v[e][0], sbf), w1 = e2m1_pack8(v[e][1], sbf);
      if (rot) {  // back to memory order
        const uint32_t t = w0;
        w0 = w1;
        w1 = t;
      }
      if (!kGuard || m < m_valid) {
        *reinterpret_cast<uint2*>(a_tile + m * kTileKBytes + ((b ^ (m & 7)) << 4) + 8 * half) = make_uint2(w0, w1);
        if (half == 0)
          sfa[((b >> 2) * kRowChunks + (m >> 7)) * kSfChunkBytes + sf_chunk_offset(m) + (b & 3)] =
              static_cast<uint8_t>(byte);
      }
    }
  }
}

// Direct activation path of the fused kernel (block_m 16 or 32, no shared
// quantization): each producer thread loads its units of a group of up to
// 4 / (BM / 16) K tiles straight from global memory -- every load of the group
// in flight at once, no staging buffer and no per-tile barrier -- then
// quantizes them into the group's stages.  The unit layout is quantize_tile's
// (unit u = tid + kThreads * e: row u / 16, 16 elements (u % 16) * 16 of the
// K tile); units past K read as zeros (as a zero-filled TMA box would), rows
// past m_valid are neither loaded nor stored.
template <int BM, int kThreads>
struct DirectTiles {
  static constexpr int kUnits = BM * 16 / kThreads;  // units per thread and K tile
  static constexpr int kGroup = 4 / kUnits;          // K tiles per group
  uint4 v[kGroup][kUnits][2];

  __device__ __forceinline__ void load(const uint8_t* a, int64_t lda_bytes, int m_base, int m_valid, int K,
                                       int kt0, int n, int tid, int M, uint32_t* err) {
    (void)M;
    (void)err;
#pragma unroll
    for (int j = 0; j < kGroup; ++j)
#pragma unroll
      for (int e = 0; e < kUnits; ++e) {
        const int u = tid + e * kThreads, m = u >> 4;
        const int col = (kt0 + j) * kTileK + (u & 15) * 16;
        v[j][e][0] = v[j][e][1] = make_uint4(0u, 0u, 0u, 0u);
        if (j < n && m < m_valid && col < K &&
            MXFP4_IN_BOUNDS(static_cast<int64_t>(m_base + m) * lda_bytes + static_cast<int64_t>(col) * 2 + 32 <=
                                static_cast<int64_t>(M) * lda_bytes,
                            err)) {
          const uint8_t* src = a + static_cast<int64_t>(m_base + m) * lda_bytes + static_cast<int64_t>(col) * 2;
          v[j][e][0] = ld_after_wait_v4(src);  // A may be the previous grid's output
          v[j][e][1] = ld_after_wait_v4(src + 16);
        }
      }
  }

  // Quantizes tile j of the group into a_tile / sfa (one stage).  The pair
  // shuffle needs both lanes of a block: a warp's units are skipped only when
  // both of its rows are past m_valid (warp-uniform).
  __device__ __forceinline__ void quantize(int j, uint8_t* a_tile, uint8_t* sfa, int tid, int m_valid) const {
    const int pw = tid >> 5, half = tid & 1;
#pragma unroll
    for (int e = 0; e < kUnits; ++e) {
      if (2 * pw + 16 * e >= m_valid) continue;  // warp-uniform
      const int u = tid + e * kThreads;
      const int m = u >> 4, b = (u >> 1) & 7;
      uint32_t amax = absmax16_bf16(v[j][e][0], v[j][e][1]);
      amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      const uint32_t byte = scale_byte_from_amax(amax);
      const uint16_t sbf = scale_bf16_from_byte(byte);
      const uint32_t w0 = e2m1_pack8(v[j][e][0], sbf), w1 = e2m1_pack8(v[j][e][1], sbf);
      if (m < m_valid) {
        *reinterpret_cast<uint2*>(a_tile + m * kTileKBytes + ((b ^ (m & 7)) << 4) + 8 * half) = make_uint2(w0, w1);
        if (half == 0) sfa[(b >> 2) * kSfChunkBytes + sf_chunk_offset(m) + (b & 3)] = static_cast<uint8_t>(byte);
      }
    }
  }
};

// The same quantization for a tile shared along N: the tile's codes and the
// scale words of its rows go to the same stage of every CTA that shares it
// (`share` CTAs, cluster ranks rank0 + rank_step * t), by st.async completing
// on that CTA's full_a barrier of the stage -- the receiver waits for
// rows_valid x 136 bytes (128 of codes, two 4-byte scale words).  A scale word
// holds the four blocks of one 128-wide chunk of a row: in a half-warp (one
// row), lanes 8c + 2j hold block 4c + j, gathered by four shuffles.
template <int BM, int kThreads, int kRowChunks>
__device__ __forceinline__ void quantize_tile_push(const uint8_t* abf, uint32_t a_tile_s, uint32_t sfa_s,
                                                   uint32_t bar_s, int tid, int rows_valid, int share,
                                                   uint32_t rank0, uint32_t rank_step) {
  constexpr int kUnits = BM * 16 / kThreads;
  const int lane = tid & 31, pw = tid >> 5;
  const int rot = (lane >> 2) & 1;
  const int half = lane & 1;
  constexpr int kBatch = kUnits < (BM < 128 ? 4 : 2) ? kUnits : (BM < 128 ? 4 : 2);
#pragma unroll(BM < 256 ? kUnits / kBatch : 1)
  for (int k0 = 0; k0 < kUnits; k0 += kBatch) {
    uint4 v[kBatch][2];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const uint8_t* src = abf + (tid + (k0 + e) * kThreads) * 32;
      if (2 * pw + 16 * (k0 + e) < rows_valid) {
        v[e][0] = *reinterpret_cast<const uint4*>(src + 16 * rot);
        v[e][1] = *reinterpret_cast<const uint4*>(src + 16 * (rot ^ 1));
      }
    }
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      if (2 * pw + 16 * (k0 + e) >= rows_valid) continue;  // warp-uniform (rows come in pairs)
      const int u = tid + (k0 + e) * kThreads;
      const int m = u >> 4, b = (u >> 1) & 7;
      uint32_t amax = absmax16_bf16(v[e][0], v[e][1]);
      amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      const uint32_t byte = scale_byte_from_amax(amax);
      const uint16_t sbf = scale_bf16_from_byte(byte);
      uint32_t w0 = e2m1_pack8(v[e][0], sbf), w1 = e2m1_pack8(v[e][1], sbf);
      if (rot) {
        const uint32_t t = w0;
        w0 = w1;
        w1 = t;
      }
      const int base = lane & ~7;
      const uint32_t word = __shfl_sync(0xFFFFFFFFu, byte, base) | (__shfl_sync(0xFFFFFFFFu, byte, base + 2) << 8) |
                            (__shfl_sync(0xFFFFFFFFu, byte, base + 4) << 16) |
                            (__shfl_sync(0xFFFFFFFFu, byte, base + 6) << 24);
      const uint32_t code_off = a_tile_s + m * kTileKBytes + ((b ^ (m & 7)) << 4) + 8 * half;
      const uint32_t sf_off = sfa_s + ((b >> 2) * kRowChunks + (m >> 7)) * kSfChunkBytes + sf_chunk_offset(m);
      for (int t = 0; t < share; ++t) {
        const uint32_t r = rank0 + rank_step * static_cast<uint32_t>(t);
        const uint32_t cbar = map_to_rank(bar_s, r);
        st_async_v2(map_to_rank(code_off, r), w0, w1, cbar);
        if ((lane & 7) == 0) st_async_b32(map_to_rank(sf_off, r), word, cbar);
      }
    }
  }
}

// kHostC: every element of C is also written to args.c_host (mapped host
// memory); a separate instantiation, so the common kernels carry none of it.
// kShare (fused only): the args.share CTAs of a cluster that hold neighbouring
// N tiles of the same rows and K split quantize the split's K tiles between
// them -- tile i by the CTA of share rank i % share -- and push each tile's
// codes and scales into all of their operand buffers (quantize_tile_push).
// The cluster is splits x share; every stage holds its own K tile (stages ==
// K tiles per split), so nothing is refilled.
template <int BM, bool kFused, bool kHostC, bool kShare>
__global__ void __launch_bounds__(TileCfg<BM, kFused>::kThreads, 2)
    mxfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_c, const GemmArgs args) {
  using C = TileCfg<BM, kFused>;
  // fused, block_m <= 32, not shared: activation straight from global memory
  // into registers (DirectTiles); otherwise by TMA into shared memory
  constexpr bool kDirect = kFused && !kShare && BM <= 32;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int stages = args.stages;
  // activation buffers: the fused kernel's bf16 staging ring (abf_ring
  // buffers, tile i in buffer i % abf_ring, free again once quantized) is
  // separate from the stages; the unfused kernel's codes land in the stages
  const int nbuf = max(stages, args.abf_ring);
  auto full_w = [&](int s) { return sbase + args.bar_off + 8u * s; };                 // weight codes + scales
  auto full_a = [&](int s) { return sbase + args.bar_off + 8u * (stages + s); };      // operand ready for the MMA
  auto empty = [&](int s) { return sbase + args.bar_off + 8u * (2 * stages + s); };   // stage consumed
  auto full_in = [&](int r) { return sbase + args.bar_off + 8u * (3 * stages + r); }; // activation buffer (TMA)
  auto abf_free = [&](int r) { return sbase + args.bar_off + 8u * (3 * stages + nbuf + r); };
  const uint32_t accum_bar = sbase + args.bar_off + 8u * (3 * stages + 2 * nbuf);
  // split-K: counts the bytes of the peers' partial blocks this CTA owns
  const uint32_t red_bar = accum_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + args.bar_off + 8 * (3 * stages + 2 * nbuf + 2));
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int splits = args.splits;
  // K split of this CTA = its x in the cluster; with kShare, its share rank is y
  const uint32_t rank = (splits > 1 || kShare) ? cluster_ctaid_x() : 0u;
  const uint32_t share_rank = kShare ? cluster_ctaid_y() : 0u;
  const int share = kShare ? args.share : 1;
  const int n_tile = blockIdx.y, m_tile = blockIdx.z;
  const int m_base = m_tile * BM;
  const int m_valid = min(BM, args.M - m_base);
  const int valid_blocks = 4 * ((m_valid + 15) >> 4);  // 32 x 16 output blocks holding rows below M
  const int kt_begin = static_cast<int>(rank) * args.kt_per_split;
  const int kt_end = min(args.k_tiles, kt_begin + args.kt_per_split);
  const int kt_count = max(0, kt_end - kt_begin);
  // K steps (of 64) in this split's last K tile
  const int steps_last = kt_count > 0 ? min(4, (args.K - (kt_end - 1) * kTileK + 63) / 64) : 0;
  const uint64_t timeout = args.timeout_ns;
  // checked build: flat element index into C, byte range in this CTA's shared memory
  auto c_ok = [&](int64_t idx, int64_t width) {
    return MXFP4_IN_BOUNDS(idx >= 0 && idx + width <= static_cast<int64_t>(args.M) * args.N, args.err);
  };
  auto smem_ok = [&](uint32_t off, uint32_t bytes) { return MXFP4_IN_BOUNDS(off + bytes <= args.smem_total, args.err); };
  (void)c_ok;
  (void)smem_ok;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_b);
    prefetch_tmap(&tmap_a);
    if (args.c_tma) prefetch_tmap(&tmap_c);
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_w(s), 1);
      // fused: one arrival per producer warp (kShare: its own arrival + the
      // pushed bytes); unfused: the producer warps' scale arrivals plus the
      // codes' TMA (its arrival + bytes), so the MMA issuer waits on one barrier
      mbar_init(full_a(s), kShare ? 1 : kFused ? C::kAWarps : C::kAWarps + 1);
      mbar_init(empty(s), 1);
    }
    if constexpr (kShare) {
      // every stage's operand arrives from the CTA that quantizes its K tile:
      // arm each with the bytes it will receive (a_box_rows x 136)
      for (int s = 0; s < kt_count && s < stages; ++s)
        mbar_arrive_expect_tx(full_a(s), args.a_box_rows * (kTileKBytes + 8));
      // (the host gives a shared plan a stage per K tile and a bf16 buffer per own tile)
      if (kt_count > stages || (kt_count + args.share - 1) / args.share > args.abf_ring) {
        report_error(args.err, kErrBadPlan);
        *abort_flag = 1u;
      }
    }
    for (int r = 0; r < nbuf; ++r) {
      mbar_init(full_in(r), 1);
      mbar_init(abf_free(r), C::kAWarps);
    }
    mbar_init(accum_bar, 1);
    // split-K: armed with the bytes of the (splits - 1) peer partials of each
    // block this CTA owns (blocks bi = rank, rank + splits, ... below valid_blocks)
    if (splits > 1) {
      mbar_init(red_bar, 1);
      const int owned = (valid_blocks - static_cast<int>(rank) + splits - 1) / splits;
      if (owned > 0) mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>(owned * (splits - 1) * kBlockBytes));
    }
    *abort_flag = 0u;
    fence_mbar_init();
    if (kFused && args.weights_early) {
      // fused: the weights of the first stages, issued by the thread that has
      // just initialised their barriers, before the CTA's set-up (tensor
      // memory, CTA barrier) rather than after it: they are the first operand
      // the call waits for when it starts just ahead of its grid wait.  (The
      // pre-quantized kernel keeps them behind its set-up: issued earlier they
      // compete with the quantize pass that runs just before it, 6.03 -> 6.20
      // us per call at M=64.)
      const uint64_t policy_w = policy_evict_first();
      for (int i = 0; i < stages && i < kt_count; ++i) {
        const int kt = kt_begin + i;
        const uint32_t bar = full_w(i);
        mbar_arrive_expect_tx(bar, C::kBTileBytes + kSfTileBytes);
        tma_load_2d(sbase + i * C::kBTileBytes, &tmap_b, kt * kTileKBytes, n_tile * kTileN, bar, policy_w);
        bulk_load(sbase + args.sfw_off + i * kSfTileBytes,
                  args.b_sf + (static_cast<size_t>(n_tile) * args.k_tiles + kt) * kSfTileBytes, kSfTileBytes, bar,
                  policy_w);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), args.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  // Peers push into this CTA's buffers and barriers only after every CTA of
  // the cluster has initialised its barriers: kShare waits here (its pushes
  // start in the main loop); a K split arrives now and waits just before its
  // epilogue pushes, by when every peer has long arrived.
  if constexpr (kShare) {
    cluster_sync_all();
  } else {
    if (splits > 1) cluster_arrive_release();
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int nacc = args.accumulators;                 // independent accumulators (1, 2 or 4)
  const uint32_t tmem_sf = tmem_base + nacc * BM;     // scale columns follow the accumulators

  // The next call in the stream may start its own prologue now (or, with
  // trigger_late, once this grid's activation loads are under way: at most
  // one grid ahead, and its prologue's weight loads do not queue in front of
  // this grid's activation loads).  Reads of data an earlier grid may write (the activation) and
  // every global write come after grid_dependency_wait(); before it, only the
  // weights (read-only for the lifetime of the call, by contract) and L2
  // prefetches.
  if (!args.trigger_late) grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp runs the loop, so waits, addresses and coordinates stay
    // warp-uniform; one elected lane issues the copies.
    const bool leader = elect_one();
    const uint64_t policy_b = policy_evict_first();  // weights: read once per call
    const uint64_t policy_a = policy_evict_last();   // activations: shared by every N tile
    const int pre = min(stages, kt_count);
    // K tile i of this split into stage s
    auto issue_w = [&](int i, int s) {
      const int kt = kt_begin + i;
      const uint32_t bar = full_w(s), dst_b = sbase + s * C::kBTileBytes, dst_sf = sbase + args.sfw_off + s * kSfTileBytes;
      const uint8_t* src_sf = args.b_sf + (static_cast<size_t>(n_tile) * args.k_tiles + kt) * kSfTileBytes;
      if (leader) {
        mbar_arrive_expect_tx(bar, C::kBTileBytes + kSfTileBytes);
        tma_load_2d(dst_b, &tmap_b, kt * kTileKBytes, n_tile * kTileN, bar, policy_b);
        bulk_load(dst_sf, src_sf, kSfTileBytes, bar, policy_b);
      }
    };
    // activation tile i: fused into bf16 staging buffer s = i % abf_ring,
    // unfused into stage s
    auto issue_a = [&](int i, int s) {
      const int kt = kt_begin + i;
      const uint32_t bar = kFused ? full_in(s) : full_a(s);
      if constexpr (kFused) {
        const uint32_t dst = sbase + args.abf_off + s * args.abf_stage_bytes;
        if (leader) {
          mbar_arrive_expect_tx(bar, args.a_box_rows * kTileK * 2);
          tma_load_2d(dst, &tmap_a, kt * kTileK, m_base, bar, policy_a);
        }
      } else {
        const uint32_t dst = sbase + args.a_off + s * C::kATileBytes;
        if (leader) {
          mbar_arrive_expect_tx(bar, args.a_box_rows * kTileKBytes);
          tma_load_2d(dst, &tmap_a, kt * kTileKBytes, m_base, bar, policy_a);
        }
      }
    };
    if (args.weights_early) {
      if constexpr (!kFused)
        for (int i = 0; i < pre; ++i) issue_w(i, i);  // (fused: thread 0 issued them during set-up)
    } else {
      for (int i = 0; i < kt_count; ++i) {
        const int kt = kt_begin + i;
        const uint8_t* src_sf = args.b_sf + (static_cast<size_t>(n_tile) * args.k_tiles + kt) * kSfTileBytes;
        if (leader) {
          tma_prefetch_l2_2d(&tmap_b, kt * kTileKBytes, n_tile * kTileN);
          bulk_prefetch_l2(src_sf, kSfTileBytes);
        }
      }
    }
    for (int i = 0; i < kt_count; ++i) {
      const int x = kFused ? (kt_begin + i) * kTileK : (kt_begin + i) * kTileKBytes;
      if (leader) tma_prefetch_l2_2d(&tmap_a, x, m_base);
    }
    grid_dependency_wait();
    if (!args.weights_early)
      for (int i = 0; i < pre; ++i) issue_w(i, i);
    const int ring_a = kFused ? args.abf_ring : stages;  // activation buffers
    // kShare: this CTA loads (and quantizes) only K tiles share_rank, + share, ...
    const int own = kDirect ? 0 : kShare ? (kt_count - static_cast<int>(share_rank) + share - 1) / share : kt_count;
    const int pre_a = min(ring_a, own);
    if constexpr (kShare) {
      for (int j = 0; j < pre_a; ++j) issue_a(static_cast<int>(share_rank) + j * share, j);
    } else {
      for (int i = 0; i < pre_a; ++i) issue_a(i, i);
    }
    // (direct path: the producers trigger, once their loads have landed)
    if (args.trigger_late && !kDirect) grid_launch_dependents();
    int issued_w = pre, issued_a = pre_a;
    // refills: a stage's weights once its MMAs are done; an activation buffer
    // once its tile is quantized (fused) or with its stage (unfused).  The
    // ring and the stages differ in size, so a tile may need either or both.
    // (kShare: the ring holds every own tile and the stages every tile.)
    for (int i = kShare ? kt_count : min(pre, pre_a); i < kt_count; ++i) {
      bool ok = true;
      if (i >= pre) {
        const int s = i % stages, round = i / stages;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(empty(s), (round - 1) & 1, timeout));
        if (!ok) {
          if (leader) report_error(args.err, kErrWaitEmpty);
          *abort_flag = 1u;
        }
        if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) break;
        issue_w(i, s);
        issued_w = i + 1;
      }
      if (kDirect || i < pre_a) continue;
      if constexpr (kFused) {
        const int r = i % ring_a, round_a = i / ring_a;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(abf_free(r), (round_a - 1) & 1, timeout));
        if (!ok) {
          if (leader) report_error(args.err, kErrWaitEmpty);
          *abort_flag = 1u;
        }
        if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) break;
        issue_a(i, r);
      } else {
        issue_a(i, i % stages);
      }
      issued_a = i + 1;
    }
    // Before the CTA can exit, every copy it issued must have landed.
    for (int s = 0; s < stages && s < issued_w; ++s) {
      const uint32_t parity = ((s + stages * ((issued_w - 1 - s) / stages)) / stages) & 1;
      if (!mbar_wait(full_w(s), parity, timeout) && leader) report_error(args.err, kErrWaitDrain);
    }
    for (int r = 0; r < ring_a && r < issued_a; ++r) {
      const uint32_t parity = ((r + ring_a * ((issued_a - 1 - r) / ring_a)) / ring_a) & 1;
      if (!mbar_wait(kFused ? full_in(r) : full_a(r), parity, timeout) && leader) report_error(args.err, kErrWaitDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // One elected lane runs the whole role: it waits on the barriers, issues
    // the tcgen05 copies and MMAs, and issues every commit (a commit tracks
    // the issuing thread's earlier operations).  No warp votes or warp
    // barriers on the per-tile path; the other lanes wait at the end.
    if (elect_one()) {
      bool triggered = !args.trigger_late;
      // Weight scales of stage s to tensor memory once the stage's weights
      // have landed; false if the wait gave up.
      auto weight_scales = [&](int s, int round) {
        if (!mbar_wait(full_w(s), round & 1, timeout)) {
          report_error(args.err, kErrWaitTma);
          *abort_flag = 1u;
        }
        if (*abort_flag != 0u) return false;
        tc_fence_after_sync();
        const uint32_t sfw_t = tmem_sf + s * C::kSfCols;  // weight scales: 2 chunks x 4 columns
        const uint32_t sfw_s = sbase + args.sfw_off + s * kSfTileBytes;
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_cp_32x128b_warpx4(sfw_t + 4 * c, smem_desc(sfw_s + c * kSfChunkBytes, 128, 128, 0));
        return true;
      };
      // The stages loaded first hold weights that arrive before the activation
      // (under programmatic launch, before the previous grid has finished): their
      // scales go to tensor memory up front, off the activation's critical path.
      const int pre = min(stages, kt_count);
      uint32_t mma_a_off = args.a_off, mma_sfa_off = args.sfa_off;
      int mma_k = args.K;
      asm volatile("" : "+r"(mma_a_off), "+r"(mma_sfa_off), "+r"(mma_k));  // parameters read before the waits
      bool alive = true;
      // weights loaded after the grid wait arrive stage by stage: copy only the
      // first stage's scales up front and each later one just before its tile,
      // so tile 0 never waits for the last stage's weights
      const int pre_copy = args.weights_early ? pre : min(pre, 1);
      for (int i = 0; i < pre_copy && alive; ++i) alive = weight_scales(i, 0);
      // stage 0's descriptors; stage s adds s tiles (the address field counts 16-byte units)
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(sbase + mma_a_off, 16, 1024, 2);
      const uint32_t sfa_s0 = sbase + mma_sfa_off;
      for (int i = 0, s = 0, round = 0; i < kt_count && alive; ++i, s = s + 1 < stages ? s + 1 : 0, round += s == 0) {
        const uint32_t sfw_t = tmem_sf + s * C::kSfCols;
        const uint32_t sfa_t = sfw_t + 8;                 // activation scales: 2 x kRowChunks x 4
        const uint32_t sfa_s = sfa_s0 + s * C::kSfaStageBytes;
        const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(s * (C::kBTileBytes >> 4));
        const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(s * (C::kATileBytes >> 4));
        const int k0 = (kt_begin + i) * kTileK;
        if (i >= pre_copy && !weight_scales(s, round)) break;  // a later or reloaded stage
        // (another role's abort shows up here as a wait that runs out)
        if (!mbar_wait(full_a(s), round & 1, timeout)) {
          report_error(args.err, kErrWaitA);
          *abort_flag = 1u;
          break;
        }
        if (!triggered) {  // the activation has landed: the next grid may start
          grid_launch_dependents();
          triggered = true;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < 2 * C::kRowChunks; ++c)
          tmem_cp_32x128b_warpx4(sfa_t + 4 * c, smem_desc(sfa_s + c * kSfChunkBytes, 128, 128, 0));
        if (nacc == 1 && k0 + kTileK <= mma_k) {
          // a whole K tile into the one accumulator: four MMAs whose operands
          // differ only by compile-time offsets (the issuing lane's own
          // instruction stream sets the MMA rate at these tile sizes)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_mxf4(tmem_base, a_desc + 2 * j, b_desc + 2 * j, mxf4_idesc<BM>((j & 1) * 2), sfw_t + 4 * (j >> 1),
                     sfa_t + 4 * C::kRowChunks * (j >> 1), (i | j) != 0);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (k0 + 64 * j >= mma_k) break;
            const uint32_t sid = (j & 1) * 2;
            // +32 bytes of K per step inside the 128-byte swizzle row (>> 4 -> +2)
            // K step g = 4i + j accumulates into tile g % nacc: nacc independent
            // chains the tensor core can overlap (summed in the epilogue)
            const int g = 4 * i + j, acc = g & (nacc - 1);
            mma_mxf4(tmem_base + acc * BM, a_desc + 2 * j, b_desc + 2 * j, mxf4_idesc<BM>(sid), sfw_t + 4 * (j >> 1),
                     sfa_t + 4 * C::kRowChunks * (j >> 1), g >= nacc);
          }
        }
        if (i + stages < kt_count) tc_commit(empty(s));  // frees the stage when these MMAs finish
      }
      tc_commit(accum_bar);  // always: the epilogue waits on it
      if (!triggered) grid_launch_dependents();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ activation producer
    const int tid = threadIdx.x - 64;
    // the kernel arguments the loop reads, fetched before the wait (a first
    // read of a parameter can miss the constant cache)
    uint32_t a_off = args.a_off, sfa_off = args.sfa_off, abf_off = args.abf_off;
    uint32_t abf_stage_bytes = args.abf_stage_bytes;
    int c_tma = args.c_tma;  // (for the epilogue)
    int ring_a = kFused ? args.abf_ring : 1;
    asm volatile("" : "+r"(a_off), "+r"(sfa_off), "+r"(abf_off), "+r"(abf_stage_bytes), "+r"(c_tma), "+r"(ring_a));
    bool triggered = !args.trigger_late;
    grid_dependency_wait();  // the activation (and C) may belong to the earlier grid
    const int64_t nblk = args.K / 32;
    // unfused: the 8 scale bytes of row `tid` for K tile i (one row per thread;
    // block_m <= 256 = the producer thread count): one 8-byte load when rows
    // are 8-byte aligned (K a multiple of 256), else byte by byte
    const bool scales_vec8 = nblk % 8 == 0 && (reinterpret_cast<uintptr_t>(args.a_scales) & 7u) == 0;
    auto load_scales = [&](int i, uint32_t& w0, uint32_t& w1) {
      const int64_t j0 = static_cast<int64_t>(kt_begin + i) * 8;
      const uint8_t* src = args.a_scales + static_cast<int64_t>(m_base + tid) * nblk + j0;
      if (!MXFP4_IN_BOUNDS(static_cast<int64_t>(m_base + tid) * nblk + j0 < static_cast<int64_t>(args.M) * nblk,
                           args.err)) {
        w0 = w1 = 0u;
        return;
      }
      if (scales_vec8) {
        const uint2 v = ld_after_wait_v2(src);  // written by the quantize pass before this grid
        w0 = v.x;
        w1 = v.y;
        return;
      }
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int jb = 0; jb < 8; ++jb)
        if (j0 + jb < nblk) w[jb >> 2] |= ld_after_wait_u8(src + jb) << (8 * (jb & 3));
      w0 = w[0];
      w1 = w[1];
    };
    constexpr int kPreK = kFused ? 1 : 8;
    uint32_t sc_pre[kPreK][2];
    if constexpr (!kFused) {
      if (tid < m_valid) {
#pragma unroll
        for (int i = 0; i < kPreK; ++i)
          if (i < kt_count) load_scales(i, sc_pre[i][0], sc_pre[i][1]);
      }
    }
    if constexpr (kShare) {
      // quantize this CTA's own K tiles, each into the same stage of every
      // CTA sharing it; the MMA warps wait on their own barriers
      const int own = (kt_count - static_cast<int>(share_rank) + share - 1) / share;
      const uint32_t rank0 = rank;  // share rank t is cluster rank rank + splits * t
      for (int j = 0; j < own; ++j) {
        const int i = static_cast<int>(share_rank) + j * share;
        if (!*abort_flag && !mbar_wait(full_in(j), 0, timeout)) {
          report_error(args.err, kErrWaitTma);
          *abort_flag = 1u;
        }
        if (!triggered) {  // the activation tile has landed: the next grid may start
          grid_launch_dependents();
          triggered = true;
        }
        if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) break;
        quantize_tile_push<BM, C::kAThreads, C::kRowChunks>(
            smem + abf_off + j * abf_stage_bytes, sbase + a_off + i * C::kATileBytes,
            sbase + sfa_off + i * C::kSfaStageBytes, full_a(i), tid, args.a_box_rows, share, rank0,
            static_cast<uint32_t>(splits));
      }
    }
    if constexpr (kDirect) {
      // groups of DirectTiles::kGroup K tiles (at most one per stage): the
      // group's loads first, then, stage by stage, wait until the stage is
      // free, quantize into it and hand it to the MMA warp
      using D = DirectTiles<BM, C::kAThreads>;
      const int group = min(D::kGroup, stages);
      const uint8_t* a_glob = static_cast<const uint8_t*>(args.a);
      int64_t lda_bytes = args.lda * 2;
      int kdim = args.K;
      asm volatile("" : "+l"(a_glob), "+l"(lda_bytes), "+r"(kdim));
      D tiles;
      int s = 0, round = 0;  // stage and reuse round of the next K tile
      for (int g0 = 0; g0 < kt_count; g0 += group) {
        const int n = min(group, kt_count - g0);
        tiles.load(a_glob, lda_bytes, m_base, m_valid, kdim, kt_begin + g0, n, tid, args.M, args.err);
        if (!triggered) {  // this grid's activation loads are under way: the next grid may start
          grid_launch_dependents();
          triggered = true;
        }
        bool stop = false;
#pragma unroll
        for (int j = 0; j < D::kGroup; ++j) {
          if (j >= n) break;
          if (round > 0) {  // a reused stage: wait until its MMAs are done
            if (!*abort_flag && !mbar_wait(empty(s), (round - 1) & 1, timeout)) {
              report_error(args.err, kErrWaitEmpty);
              *abort_flag = 1u;
            }
            stop = __any_sync(0xFFFFFFFFu, *abort_flag != 0u);  // warp-uniform: the shuffles need every lane
            if (stop) break;
          }
          tiles.quantize(j, smem + a_off + s * C::kATileBytes, smem + sfa_off + s * C::kSfaStageBytes, tid, m_valid);
          fence_proxy_async_smem();  // this thread's generic stores, visible to tcgen05
          __syncwarp();
          if (lane == 0) mbar_arrive(full_a(s));
          if (++s == stages) {
            s = 0;
            ++round;
          }
        }
        if (stop) break;
      }
    }
    for (int i = 0, s = 0, round = 0, r = 0, round_a = 0; !kShare && !kDirect && i < kt_count;
         ++i, s = s + 1 < stages ? s + 1 : 0, round += s == 0, r = r + 1 < ring_a ? r + 1 : 0, round_a += r == 0) {
      if (round > 0 && !mbar_wait(empty(s), (round - 1) & 1, timeout)) {
        report_error(args.err, kErrWaitEmpty);
        *abort_flag = 1u;
      }
      // fused: the tile's bf16 buffer r.  Unfused: nothing to wait for -- the
      // codes' TMA completes on full_a(s) itself, beside these warps' scales.
      if (kFused && !*abort_flag && !mbar_wait(full_in(r), round_a & 1, timeout)) {
        report_error(args.err, kErrWaitTma);
        *abort_flag = 1u;
      }
      if (!triggered) {  // fused: the activation tile has landed; the next grid may start
        grid_launch_dependents();
        triggered = true;
      }
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0u)) break;  // warp-uniform: the shuffles below need every lane
      uint8_t* a_tile = smem + a_off + s * C::kATileBytes;
      uint8_t* sfa = smem + sfa_off + s * C::kSfaStageBytes;
      if constexpr (kFused) {
        const uint8_t* abf = smem + abf_off + r * abf_stage_bytes;
        if (m_valid >= BM)
          quantize_tile<BM, C::kAThreads, C::kRowChunks, false>(abf, a_tile, sfa, tid, m_valid);
        else
          quantize_tile<BM, C::kAThreads, C::kRowChunks, true>(abf, a_tile, sfa, tid, m_valid);
      } else {
        // Pre-quantized activation: the codes arrived by TMA; place the
        // natural [M, K/32] scales into the chunk layout, one row per thread
        // (loaded for the first kPreK tiles before the loop, see below).
        if (tid < m_valid) {
          uint32_t w0, w1;
          if (i < kPreK) {
            w0 = w1 = 0u;
#pragma unroll
            for (int pk = 0; pk < kPreK; ++pk)  // register select (no dynamic indexing)
              if (pk == i) {
                w0 = sc_pre[pk][0];
                w1 = sc_pre[pk][1];
              }
          } else {
            load_scales(i, w0, w1);
          }
          const int r = tid;
          *reinterpret_cast<uint32_t*>(sfa + (0 * C::kRowChunks + (r >> 7)) * kSfChunkBytes + sf_chunk_offset(r)) = w0;
          *reinterpret_cast<uint32_t*>(sfa + (1 * C::kRowChunks + (r >> 7)) * kSfChunkBytes + sf_chunk_offset(r)) = w1;
        }
      }
      fence_proxy_async_smem();  // make this thread's generic stores visible to tcgen05
      __syncwarp();              // ... and ordered before the warp's single arrival
      if (lane == 0) {
        mbar_arrive(full_a(s));
        if constexpr (kFused) mbar_arrive(abf_free(r));  // the bf16 buffer may be refilled
      }
    }

    if (!triggered) grid_launch_dependents();
    // ------------------------------------------------------------------ epilogue
    const bool ok = mbar_wait(accum_bar, 0, timeout);
    if (!ok) report_error(args.err, kErrWaitAccum);
    tc_fence_after_sync();
    const bool have = ok && kt_count > 0 && !*abort_flag;
    if (!kShare && splits > 1) cluster_wait_acquire();  // every peer's barriers are initialised
    const int qr = warp & 3;           // TMEM lanes this warp may read
    const int h = (warp - 2) >> 2;     // which half of the column chunks
    const int chunks = (m_valid + 15) >> 4;
    if (splits == 1 && c_tma && chunks == 1 && nacc == 1) {
      // one 16-row chunk (block_m 16, or M <= 16): both warp halves load it,
      // each converts and stages 8 of its rows, so all eight epilogue warps work
      uint32_t r[16];
      if (have) {
        tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(qr * 32) << 16), r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = 0u;
      }
      __nv_bfloat16* cs = reinterpret_cast<__nv_bfloat16*>(smem) + (h * 8) * kTileN + qr * 32 + lane;
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint32_t lo = h ? r[8 + e] : r[e], hi = h ? r[9 + e] : r[e + 1];
        const __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
        cs[e * kTileN] = pr.x;
        cs[(e + 1) * kTileN] = pr.y;
      }
    } else
#pragma unroll 1
    for (int c = h; c < chunks; c += 2) {
      uint32_t r[16];
      if (have) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(qr * 32) << 16) + c * 16;
        tmem_ld_32x32b_x16(taddr, r);
        // accumulators that received no K step (fewer steps than tiles) are skipped
        const int used = min(nacc, 4 * (kt_count - 1) + steps_last);
        for (int a = 1; a < used; ++a) {
          uint32_t t[16];
          tmem_ld_32x32b_x16(taddr + a * BM, t);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(t[e]));
        }
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = 0u;
      }
      if (splits == 1 && c_tma) {
        // no K split: bf16 into the output tile [BM rows][128 columns] at
        // offset 0 (lane = column n, register e = row m, rows e and e + 1
        // converted as one pair; a warp's stores of one row are 64 contiguous
        // bytes), sent by one TMA store below
        __nv_bfloat16* cs = reinterpret_cast<__nv_bfloat16*>(smem) + (c * 16) * kTileN + qr * 32 + lane;
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(r[e]), __uint_as_float(r[e + 1]));
          cs[e * kTileN] = pr.x;
          cs[(e + 1) * kTileN] = pr.y;
        }
        continue;
      }
      if (splits == 1) {
        // no K split and no TMA store (N not a multiple of 8): bf16 straight
        // from the accumulator registers to C
        const int n = n_tile * kTileN + qr * 32 + lane;
        if (n < args.N) {
          __nv_bfloat16* col = args.c + static_cast<int64_t>(m_base) * args.N + n;
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (c * 16 + e < m_valid && c_ok((static_cast<int64_t>(m_base) + c * 16 + e) * args.N + n, 1))
              col[static_cast<int64_t>(c * 16 + e) * args.N] = __float2bfloat16_rn(__uint_as_float(r[e]));
          if constexpr (kHostC) {
            __nv_bfloat16* hcol = args.c_host + static_cast<int64_t>(m_base) * args.N + n;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c * 16 + e < m_valid && c_ok((static_cast<int64_t>(m_base) + c * 16 + e) * args.N + n, 1))
                hcol[static_cast<int64_t>(c * 16 + e) * args.N] = __float2bfloat16_rn(__uint_as_float(r[e]));
          }
        }
        continue;
      }
      // K split: block (chunk c of 16 activation rows, lane quarter qr) goes
      // to cluster rank (4c + qr) % splits, into that CTA's slot
      // [this rank][(4c + qr) / splits], by st.async counted on the owner's
      // red_bar (the owner waits for its bytes; no cluster barrier).  The
      // staging area is separate from the stage buffers, so a peer still
      // running its MMAs is never disturbed.
      const int bi = 4 * c + qr;
      const uint32_t owner = static_cast<uint32_t>(bi % splits);
      const uint32_t dst = sbase + args.stg_off +
                           (static_cast<uint32_t>(rank) * args.stg_blocks + bi / splits) * kBlockBytes + lane * 4;
      if (owner == rank) {  // this CTA's own blocks: plain shared-memory stores
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (smem_ok(dst - sbase + e * 128, 4)) *reinterpret_cast<float*>(smem + (dst - sbase) + e * 128) = __uint_as_float(r[e]);
      } else {
        const uint32_t peer = owner + static_cast<uint32_t>(splits) * share_rank;
        const uint32_t cdst = map_to_rank(dst, peer), cbar = map_to_rank(red_bar, peer);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (smem_ok(dst - sbase + e * 128, 4)) st_async_b32(cdst + e * 128, r[e], cbar);
      }
    }
    if (splits == 1 && c_tma) {
      fence_proxy_async_smem();        // the tile's generic stores, visible to the TMA engine
      named_barrier(1, C::kAThreads);  // every epilogue warp has written its part
      if (tid == 0) {
        tma_store_2d(&tmap_c, n_tile * kTileN, m_base, sbase);
        bulk_commit_group();
      }
      if constexpr (kHostC) {
        // the host copy of the tile, read back from shared memory 16 bytes at
        // a time: row m, 8 columns per chunk (N % 8 == 0 here, so a chunk is
        // wholly inside or wholly past N), 256 contiguous bytes per row
        const int n_base = n_tile * kTileN;
        for (int it = tid; it < m_valid * 16; it += C::kAThreads) {
          const int m = it >> 4, n = n_base + (it & 15) * 8;
          if (n < args.N && c_ok(static_cast<int64_t>(m_base + m) * args.N + n, 8))
            *reinterpret_cast<uint4*>(args.c_host + static_cast<int64_t>(m_base + m) * args.N + n) =
                *reinterpret_cast<const uint4*>(smem + (m * kTileN + (it & 15) * 8) * 2);
        }
      }
    }
  }

  // ---------------------------------------------------------------------- every partial delivered
  // The parameters the K-split sum reads, fetched before the barrier (a first
  // read of a kernel parameter can miss the constant cache); the empty asm
  // makes each value live here, so the loads are not sunk past the barrier.
  int n_cols = args.N;
  __nv_bfloat16* c_out = args.c;
  uint32_t stg_stride = static_cast<uint32_t>(args.stg_blocks) * kBlockBytes;
  asm volatile("" : "+r"(n_cols), "+l"(c_out), "+r"(stg_stride));
  tc_fence_before_sync();
  if constexpr (kShare) {
    cluster_sync_all();  // no CTA leaves while a peer may still push operands into it
  } else {
    if (splits > 1 && warp < 2) cluster_wait_acquire();  // (their arrival at the start)
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, args.tmem_cols);
  }
  if (warp >= 2 && splits > 1) {
    // ------------------------------------------------ sum the owned blocks over the splits, store bf16
    // An owner waits until its peers' partials have all landed (red_bar
    // counts their bytes); its own were stored before the CTA barrier above.
    // Nothing else is waited for: a CTA that owns no block exits at once.
    const int tid = threadIdx.x - 64;
    const int mine = (valid_blocks - static_cast<int>(rank) + splits - 1) / splits;
    if (mine > 0 && !mbar_wait(red_bar, 0, timeout) && tid == 0) report_error(args.err, kErrWaitReduce);
    const int n_base = n_tile * kTileN;
    const bool vec_ok = (n_cols % 4) == 0;
    const uint32_t stg = sbase + args.stg_off;  // shared-window address: ld.shared, not generic loads
    for (int it = tid; it < mine * 128; it += C::kAThreads) {
      const int lb = it >> 7, w = it & 127, row = w >> 3, c4 = w & 7;
      const int bi = lb * splits + static_cast<int>(rank);
      const int m = (bi >> 2) * 16 + row;
      if (m >= m_valid) continue;
      const uint32_t off = lb * kBlockBytes + row * 128 + c4 * 16;
      if (!smem_ok(args.stg_off + (splits - 1) * stg_stride + off, 16)) continue;
      // every source's loads first, then the sum in rank order (deterministic)
      float4 part[kMaxSplits];
#pragma unroll
      for (int src = 0; src < kMaxSplits; ++src)
        if (src < splits) part[src] = ld_shared_f4(stg + src * stg_stride + off);
      float4 acc = part[0];
#pragma unroll
      for (int src = 1; src < kMaxSplits; ++src)
        if (src < splits) {
          acc.x += part[src].x;
          acc.y += part[src].y;
          acc.z += part[src].z;
          acc.w += part[src].w;
        }
      const int64_t gm = static_cast<int64_t>(m_base) + m;
      const int gn = n_base + (bi & 3) * 32 + c4 * 4;
      __nv_bfloat16* dst = c_out + gm * n_cols + gn;
      // columns past N are never stored: only the stored ones are checked
      if (!(gn >= n_cols || c_ok(gm * n_cols + gn, min(4, n_cols - gn)))) continue;
      if (vec_ok && gn + 3 < n_cols) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 wv;
        wv.x = *reinterpret_cast<const uint32_t*>(&lo);
        wv.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(dst) = wv;
        if constexpr (kHostC) *reinterpret_cast<uint2*>(args.c_host + gm * args.N + gn) = wv;
      } else {
        const float e[4] = {acc.x, acc.y, acc.z, acc.w};
        for (int qq = 0; qq < 4; ++qq)
          if (gn + qq < n_cols) {
            dst[qq] = __float2bfloat16_rn(e[qq]);
            if constexpr (kHostC) args.c_host[gm * args.N + gn + qq] = __float2bfloat16_rn(e[qq]);
          }
      }
    }
  }
  // the output tile must stay in shared memory until the TMA store has read it
  if (splits == 1 && args.c_tma && threadIdx.x == 64) bulk_wait_group_read0();
}

// ----------------------------------------------------------------------------- host side
template <int BM, bool kFused, bool kHostC, bool kShare>
static cudaError_t launch_t(const CUtensorMap& tmap_b, const CUtensorMap& tmap_a, const CUtensorMap& tmap_c,
                            const GemmArgs& args, const mxfp4_plan_t& plan, bool programmatic, cudaStream_t s) {
  auto kernel = mxfp4_gemm_kernel<BM, kFused, kHostC, kShare>;
  static int configured_device = -1;  // max dynamic smem (and cluster size) set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    if (kShare) {  // splits x share may exceed the portable 8
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid_x, plan.grid_y, plan.grid_z);
  cfg.blockDim = dim3(plan.threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.splits;
  attr[0].val.clusterDim.y = kShare ? plan.share : 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, tmap_b, tmap_a, tmap_c, args);
}

cudaError_t launch_gemm(const CUtensorMap& tmap_b, const CUtensorMap& tmap_a, const CUtensorMap& tmap_c,
                        const GemmArgs& args, const mxfp4_plan_t& plan, bool fused, bool programmatic,
                        cudaStream_t s) {
#define MXFP4_LAUNCH(BM_)                                                                                   \
  case BM_:                                                                                                 \
    if (args.c_host != nullptr)                                                                             \
      return fused ? launch_t<BM_, true, true, false>(tmap_b, tmap_a, tmap_c, args, plan, programmatic, s)  \
                   : launch_t<BM_, false, true, false>(tmap_b, tmap_a, tmap_c, args, plan, programmatic, s); \
    return fused ? launch_t<BM_, true, false, false>(tmap_b, tmap_a, tmap_c, args, plan, programmatic, s)   \
                 : launch_t<BM_, false, false, false>(tmap_b, tmap_a, tmap_c, args, plan, programmatic, s);
#define MXFP4_LAUNCH_SHARE(BM_)                                                                         \
  case BM_:                                                                                             \
    if (args.c_host != nullptr)                                                                         \
      return launch_t<BM_, true, true, true>(tmap_b, tmap_a, tmap_c, args, plan, programmatic, s);      \
    return launch_t<BM_, true, false, true>(tmap_b, tmap_a, tmap_c, args, plan, programmatic, s);
  if (fused && plan.share > 1) {
    switch (plan.block_m) {  // quantization shared along N: block_m up to 64
      MXFP4_LAUNCH_SHARE(16)
      MXFP4_LAUNCH_SHARE(32)
      MXFP4_LAUNCH_SHARE(64)
      default: return cudaErrorInvalidValue;
    }
  }
  switch (plan.block_m) {
    MXFP4_LAUNCH(16)
    MXFP4_LAUNCH(32)
    MXFP4_LAUNCH(64)
    MXFP4_LAUNCH(128)
    MXFP4_LAUNCH(256)
    default: return cudaErrorInvalidValue;
  }
#undef MXFP4_LAUNCH_SHARE
#undef MXFP4_LAUNCH
}

static int threads_for(int) { return 64 + 256; }

static int sf_cols_for(int bm) { return 8 + 8 * (bm > 128 ? 2 : 1); }

static uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

GemmLayout gemm_layout(int block_m, int stages, int splits, bool fused, int64_t M, int abf_ring) {
  GemmLayout L;
  const uint32_t st = static_cast<uint32_t>(stages), bm = static_cast<uint32_t>(block_m);
  L.a_off = st * kTileN * kTileKBytes;
  L.abf_off = L.a_off + st * bm * kTileKBytes;
  L.abf_stage = fused ? static_cast<uint32_t>(activation_box_rows(M, block_m)) * kTileK * 2 : 0u;
  L.abf_ring = fused ? abf_ring : 0;
  L.sfw_off = L.abf_off + static_cast<uint32_t>(L.abf_ring) * L.abf_stage;
  // without a K split the bf16 output tile is written over the operand
  // buffers once the MMAs are done: keep room for it before the scales
  if (splits == 1 && L.sfw_off < bm * kTileN * 2) L.sfw_off = bm * kTileN * 2;
  L.sfa_off = L.sfw_off + st * kSfTileBytes;
  L.stg_off = L.sfa_off + st * (bm > 128 ? 2u : 1u) * 2u * kSfChunkBytes;
  const int64_t rows = M < block_m ? M : block_m;
  const int blocks = static_cast<int>(4 * ceil_div(rows, 16));
  L.stg_blocks = splits > 1 ? static_cast<int32_t>(ceil_div(blocks, splits)) : 0;  // no split: no staging
  L.bar_off = L.stg_off + static_cast<uint32_t>(splits * L.stg_blocks) * kBlockBytes;
  const uint32_t nbuf = st > static_cast<uint32_t>(L.abf_ring) ? st : static_cast<uint32_t>(L.abf_ring);
  L.total = L.bar_off + (3 * st + 2 * nbuf + 2) * 8 + 16;  // ... accum, red_bar; tmem slot + abort flag
  return L;
}

// Shared memory one CTA of plan p requests with a bf16 ring of `ring`
// buffers; false if it exceeds the per-CTA limit.  Tensor-memory allocation
// blocks while the SM's 512 columns are taken, and a blocked CTA of one
// cluster could then wait on a CTA of another cluster that waits on it.  Each
// CTA therefore takes shared memory in proportion to its tensor-memory share
// (tmem_cols / 512 of the SM's shared memory): the CTAs that fit on an SM
// together, from any mix of these kernels, can never ask for more than 512
// columns, and no allocation ever waits.
static bool plan_smem(const mxfp4_plan_t& p, bool fused, int64_t M, const cudaDeviceProp& prop, int ring,
                      int64_t* bytes) {
  const GemmLayout L = gemm_layout(p.block_m, p.stages, p.splits, fused, M, ring);
  int64_t smem = static_cast<int64_t>(L.total) + 1024;  // + alignment slack
  const int64_t per_sm = prop.sharedMemPerMultiprocessor;
  const int64_t reserved = prop.reservedSharedMemPerBlock;
  const int64_t floor_smem = (per_sm * p.tmem_cols + 511) / 512 - reserved;
  if (smem < floor_smem) smem = floor_smem;
  smem = (smem + 15) / 16 * 16;
  *bytes = smem;
  return smem <= static_cast<int64_t>(prop.sharedMemPerBlockOptin);
}

int abf_ring_for(const mxfp4_plan_t& p, bool fused, int64_t M, const cudaDeviceProp& prop) {
  if (!fused) return 0;
  if (p.share > 1) return (p.k_tiles_per_split + p.share - 1) / p.share;  // every own tile in flight
  if (p.block_m <= 32) return 0;  // the direct path: activation loaded into registers
  // as many bf16 buffers as the split has K tiles (all in flight at once), up
  // to kAbfRing, as long as the CTA still fits -- and still shares an SM with
  // another CTA when it would with a single buffer
  auto two_per_sm = [&](int64_t smem) {
    return 2 * (smem + static_cast<int64_t>(prop.reservedSharedMemPerBlock)) <=
           static_cast<int64_t>(prop.sharedMemPerMultiprocessor);
  };
  int64_t one = 0;
  const bool fits1 = plan_smem(p, fused, M, prop, 1, &one);
  for (int r = p.k_tiles_per_split < kAbfRing ? p.k_tiles_per_split : kAbfRing; r > 1; --r) {
    int64_t b = 0;
    if (plan_smem(p, fused, M, prop, r, &b) && (!fits1 || !two_per_sm(one) || two_per_sm(b))) return r;
  }
  return 1;
}

bool finish_plan(int64_t M, int64_t N, int64_t K, bool fused, const cudaDeviceProp& prop,
                 mxfp4_plan_t* p) {
  if (p->block_m != 16 && p->block_m != 32 && p->block_m != 64 && p->block_m != 128 && p->block_m != 256)
    return false;
  const int64_t k_tiles = ceil_div(K, kTileK);
  if (p->splits < 1 || p->splits > kMaxSplits || p->splits > k_tiles) return false;
  const int64_t per = ceil_div(k_tiles, p->splits);
  // every split gets at least one K tile
  if ((p->splits - 1) * per >= k_tiles) return false;
  if (p->stages < 1 || p->stages > per) p->stages = static_cast<int32_t>(per < 6 ? per : 6);
  p->k_tiles_per_split = static_cast<int32_t>(per);
  // quantization shared along N: fused, block_m <= 64, share divides the N
  // tiles, a cluster of splits x share <= 16, and a stage per K tile
  if (p->share == 0) p->share = 1;
  if (p->share < 1) return false;
  if (p->share > 1) {
    if (!fused || p->block_m > 64 || ceil_div(N, kTileN) % p->share != 0 || p->splits * p->share > 16 ||
        p->share > per)
      return false;
    p->stages = static_cast<int32_t>(per);
  }
  p->grid_x = p->splits;
  p->grid_y = static_cast<int32_t>(ceil_div(N, kTileN));
  p->grid_z = static_cast<int32_t>(ceil_div(M, p->block_m));
  if (p->grid_y > 65535 || p->grid_z > 65535) return false;
  p->threads = threads_for(p->block_m);
  // One accumulator by default: on GB300 spreading a CTA's K steps over 2 or 4
  // independent tiles measured no faster (the MMA phase is dominated by fixed
  // start-up cost, not by the dependent chain), and it costs tensor memory.
  if (p->accumulators == 0) p->accumulators = 1;
  if (p->accumulators != 1 && p->accumulators != 2 && p->accumulators != 4) return false;
  const uint32_t tcols = pow2_at_least(p->accumulators * p->block_m + p->stages * sf_cols_for(p->block_m));
  if (tcols > 512) return false;
  p->tmem_cols = static_cast<int32_t>(tcols);
  int64_t smem = 0;
  if (!plan_smem(*p, fused, M, prop, abf_ring_for(*p, fused, M, prop), &smem)) return false;
  p->smem_bytes = static_cast<int32_t>(smem);
  return true;
}

template <int BM, bool kFused, bool kShare>
static int active_clusters_t(const mxfp4_plan_t& p) {
  auto kernel = mxfp4_gemm_kernel<BM, kFused, false, kShare>;  // the host-copy kernels use the same resources
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess) return 0;
  if (kShare && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid_x, p.grid_y, p.grid_z);
  cfg.blockDim = dim3(p.threads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.splits;
  attr[0].val.clusterDim.y = kShare ? p.share : 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error so later calls are unaffected
    return 0;
  }
  return n;
}

// How many clusters of this plan can be resident at once on the device.
static int active_clusters(const mxfp4_plan_t& p, bool fused) {
  if (fused && p.share > 1) {
    switch (p.block_m) {
      case 16: return active_clusters_t<16, true, true>(p);
      case 32: return active_clusters_t<32, true, true>(p);
      case 64: return active_clusters_t<64, true, true>(p);
      default: return 0;
    }
  }
#define MXFP4_OCC(BM_) \
  case BM_: return fused ? active_clusters_t<BM_, true, false>(p) : active_clusters_t<BM_, false, false>(p);
  switch (p.block_m) {
    MXFP4_OCC(16)
    MXFP4_OCC(32)
    MXFP4_OCC(64)
    MXFP4_OCC(128)
    MXFP4_OCC(256)
    default: return 0;
  }
#undef MXFP4_OCC
}

// The default plan.  Every call is latency-bound, so the plan minimises an
// estimate of one CTA's critical path among the plans that run in a single
// wave (every cluster resident at once, at most two CTAs per SM): each K tile
// a split runs in sequence costs ~250 ns (operand loads, tensor-memory scale
// copies, four MMAs) plus, on the fused kernel, ~200 ns per 32 activation rows
// it quantizes (so 16-row tiles halve it: at M = 32 two CTAs of 16 rows beat
// one of 32); a K split adds ~700 ns + 10 ns per row for the reduction; a
// split with more K tiles than stages adds ~1 us per reload, divided by the
// stages in flight; and a plan whose CTAs leave no room for the next call's
// beside them (twice the CTAs do not fit at the plan's CTAs per SM) adds
// ~0.5 us, the overlap the next call loses under programmatic launch
// (measured on GB300 with graph-replayed calls).  Candidates: block_m from the
// smallest tile that holds M (capped at 128; at 32 on the fused kernel up to
// M = 128) down to a quarter of it; every split count that leaves no split
// empty; 1 to 6 stages (at most the split's K tiles).  Ties prefer the larger
// block_m (fewer re-reads of the weights), then the larger stage count, then
// fewer splits.
// Plans measured best on GB300 (152 SMs) for shapes of the leaderboard where
// the estimate is not (keyed on the shape): sweeps of block_m x splits x
// stages x share, graph-replayed calls with rotating operands.  `fused` is the
// GEMM kernel's kind (the large-M shapes run the pre-quantized kernel on the
// fused entry's two-pass route).  Sharing the quantization along N is taken
// by no tuned plan: once block_m 16 and 32 load the activation straight into
// registers, the unshared plan is faster at every shape measured (16 x 3072 x
// 1536: 3.19 us against 3.73 shared); before, sharing had won there alone.
struct TunedPlan {
  int64_t M, N, K;
  bool fused;
  int block_m, splits, stages, share;
};
constexpr TunedPlan kTunedPlans[] = {
    {16, 2112, 7168, true, 16, 7, 4, 1},
    {8, 2112, 7168, true, 16, 7, 4, 1},
    {16, 3072, 1536, true, 16, 3, 2, 1},
    {256, 2880, 512, false, 64, 1, 2, 1},
    // M >= 64 with a tuned single-kernel plan: the fused entry skips the
    // two-pass route here (64 x 3072 x 1536: 4.63 us against 5.20 two-pass)
    {64, 3072, 1536, true, 32, 3, 2, 1},
    {64, 7168, 2048, false, 64, 2, 4, 1},
    {256, 3072, 1536, false, 64, 1, 6, 1},
};

bool tuned_single_kernel(int64_t M, int64_t N, int64_t K) {
  for (const TunedPlan& t : kTunedPlans)
    if (t.fused && t.M == M && t.N == N && t.K == K) return true;
  return false;
}

// Lost overlap of a plan whose CTAs leave no room for the next call's beside them, in ns.
constexpr int64_t kNoRoomNs = 500;

// Estimated critical path of one CTA, in ns (see above).
static int64_t plan_cost_ns(const mxfp4_plan_t& p, int64_t M, bool fused) {
  const int64_t rows = M < p.block_m ? M : p.block_m;
  const int64_t tile = 250 + (fused ? 200 * rows / 32 : 0);
  const int64_t tiles = p.k_tiles_per_split;
  // a stage reloaded `tiles - stages` times, each reload waiting for the MMAs
  // of the tile before it: ~1 us of load latency, shared by the stages in flight
  const int64_t refill = tiles > p.stages ? (tiles - p.stages) * 1000 / p.stages : 0;
  // a K split's reduction grows with the rows it sums: ~700 ns at 16 rows,
  // ~2 us at 128 (96x4096x1024: 4 splits of 128 rows 5.7 us, none of 64 rows 4.6)
  return tiles * tile + (p.splits > 1 ? 700 + 10 * rows : 0) + refill;
}

void default_plan(int64_t M, int64_t N, int64_t K, bool fused, const cudaDeviceProp& prop,
                  mxfp4_plan_t* p) {
  *p = mxfp4_plan_t{};
  // A tuned plan is keyed on the shape; it is taken on any device where it
  // fits and its CTAs are at most two per SM.
  for (const TunedPlan& t : kTunedPlans) {
    if (t.M != M || t.N != N || t.K != K || t.fused != fused) continue;
    mxfp4_plan_t q{};
    q.block_m = t.block_m;
    q.splits = t.splits;
    q.stages = t.stages;
    q.share = t.share;
    if (!finish_plan(M, N, K, fused, prop, &q)) continue;
    const int64_t ctas = static_cast<int64_t>(q.grid_y) * q.grid_z * q.splits;
    if (ctas <= 2 * static_cast<int64_t>(prop.multiProcessorCount)) {
      *p = q;
      return;
    }
  }
  // (block_m 256 measured slower than 128 at every M = 256 shape swept: its
  // MMAs and operand tiles cost more than the weight re-reads they save)
  // The fused kernel quantizes tiles of 16 or 32 rows straight from global
  // memory into registers; larger tiles are staged in shared memory and
  // quantized there, which measured slower up to M = 128 (65x3072x1536:
  // 32-row tiles 4.7 us, 128-row 6.6; 100x2112x1536 and 128x4096x512 also
  // fastest at 32 rows)
  int bm0 = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  if (fused && M <= 128 && bm0 > 32) bm0 = 32;
  const int64_t k_tiles = ceil_div(K, kTileK);
  const int64_t cap = 2 * static_cast<int64_t>(prop.multiProcessorCount);
  // score: one wave, then the estimate (or fewer CTAs), block_m, stages, fewer splits
  constexpr int kScore = 5;
  int64_t best[kScore] = {-1, 0, 0, 0, 0};
  for (int bm = bm0; bm >= 16 && bm * 4 >= bm0; bm /= 2) {
    for (int64_t splits = 1; splits <= kMaxSplits && splits <= k_tiles; ++splits) {
      const int64_t per = ceil_div(k_tiles, splits);
      if ((splits - 1) * per >= k_tiles) continue;  // an empty split
      for (int64_t st = 1; st <= per && st <= 6; ++st) {
        mxfp4_plan_t q{};
        q.block_m = bm;
        q.splits = static_cast<int32_t>(splits);
        q.stages = static_cast<int32_t>(st);
        if (!finish_plan(M, N, K, fused, prop, &q) || q.stages != st) continue;
        const int64_t clusters = static_cast<int64_t>(q.grid_y) * q.grid_z;
        const int64_t ctas = clusters * splits;
        const int64_t one_wave = ctas <= cap && clusters <= active_clusters(q, fused) ? 1 : 0;
        // the next call's CTAs can start beside this call's (programmatic
        // launch) when twice the CTAs fit on the device at this plan's CTAs per SM
        const int64_t per_sm =
            2 * (static_cast<int64_t>(q.smem_bytes) + prop.reservedSharedMemPerBlock) <= prop.sharedMemPerMultiprocessor
                ? 2
                : 1;
        // (a plan without that room pays ~0.5 us of lost overlap on top of its
        // estimate, rather than losing to every plan with room whatever the
        // estimates: 256x2880x7168 12.6 us with 2 splits against 16.8 without)
        const bool room_for_next = 2 * ctas <= per_sm * static_cast<int64_t>(prop.multiProcessorCount);
        const int64_t cost = plan_cost_ns(q, M, fused) + (room_for_next ? 0 : kNoRoomNs);
        const int64_t score[kScore] = {one_wave, one_wave ? -cost : -ctas, bm, st, -splits};
        bool better = false;
        for (int i = 0; i < kScore; ++i) {
          if (score[i] != best[i]) {
            better = score[i] > best[i];
            break;
          }
        }
        if (better) {
          for (int i = 0; i < kScore; ++i) best[i] = score[i];
          *p = q;
        }
      }
    }
  }
}

}  // namespace mxfp4
