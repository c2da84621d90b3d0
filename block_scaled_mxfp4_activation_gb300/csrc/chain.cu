// Several dependent MXFP4 linear layers in one persistent launch: layer l maps
// X_l [M, K_l] to C_l [M, N_l] = quant(X_l) * W_l^T, and C_l is X_{l+1}.
//
// The pages launch one quantize + GEMM (or a fused kernel) per layer and
// attribute most of each call's time to per-launch cost (submission 733989,
// "PROFILING"); a separate kernel per layer on GB300 also waits for the whole
// previous grid to finish.  Here every CTA stays resident for all layers and
// layers hand over through completion counters in global memory:
//
//   - the first layer's activation A is quantized once, cooperatively: each
//     CTA takes 16-row x 256-column units, writes their codes to the
//     workspace and their scales in the tensor-memory chunk layout, and
//     counts the unit done;
//   - every later layer's activation is quantized by the epilogue that
//     produces it: a 128-column output tile holds four whole 32-element blocks
//     of the next layer's K, so the warp owning 32 output columns reduces the
//     amax of each row's block across its lanes and writes codes and scales
//     directly (the same rule and instructions as mxfp4_quantize, applied to
//     the bf16 values stored to C_l, so the codes are bit-identical to
//     quantizing C_l separately);
//   - per CTA and K tile of a layer: warp 0 streams the weight tile (TMA,
//     128-byte swizzle) and its scales into a stage ring as soon as a stage is
//     free -- the next layer's weights load while this layer finishes; warp 10
//     waits for the activation's K tile to be complete (a counter per row tile
//     and K tile) and loads its codes (TMA, straight into the MMA operand
//     layout) and scales (bulk copy); warp 1 issues the block-scaled MMAs
//     into a tensor-memory accumulator; warps 2-9 run the epilogue;
//   - K splits (for layers with few output tiles and long K) store fp32
//     partials in the workspace; once every split of a tile has, each split
//     CTA sums a share of the tile over all partials in split order
//     (deterministic) and runs the epilogue on it;
//   - every counter returns to zero at the end of the launch (the last CTA to
//     finish clears them), so the workspace needs zeroing only once.
//
// Every wait is bounded; a wait that gives up sets the device error word and
// the CTA skips the rest of its work, still draining its copies, freeing its
// tensor memory and taking part in the final counter reset.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "tile.cuh"

namespace mxfp4 {

constexpr int kChainEpiWarps = 8;
constexpr int kChainEpiThreads = kChainEpiWarps * 32;
constexpr int kChainActWarp = 2 + kChainEpiWarps;           // warp 10: activation loads
constexpr int kChainThreads = (kChainActWarp + 1) * 32;     // 352
constexpr int kChainATileSf = 2 * kSfChunkBytes;            // activation scales per K tile (block_m <= 128)

// The item (output tile and K split) with index i of a layer.
struct ChainItem {
  int n_tile, m_tile, split, kt0, kt1;
};

__device__ __forceinline__ ChainItem chain_item(const ChainLayerArgs& L, int i) {
  ChainItem it;
  it.split = i % L.splits;
  const int t = i / L.splits;
  it.n_tile = t % L.n_tiles;
  it.m_tile = t / L.n_tiles;
  it.kt0 = it.split * L.kt_per_split;
  it.kt1 = min(L.k_tiles, it.kt0 + L.kt_per_split);
  return it;
}

template <int BM>
__global__ void __launch_bounds__(kChainThreads, 2) chain_kernel(const __grid_constant__ ChainArgs p) {
  static_assert(BM == 16 || BM == 32 || BM == 64, "block_m of the multi-layer kernel: 16, 32 or 64");
  constexpr int kATileBytes = BM * kTileKBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int stages = p.stages;
  auto full_w = [&](int s) { return sbase + p.bar_off + 8u * s; };
  auto full_in = [&](int s) { return sbase + p.bar_off + 8u * (stages + s); };
  auto empty = [&](int s) { return sbase + p.bar_off + 8u * (2 * stages + s); };
  const uint32_t accum_full = sbase + p.bar_off + 8u * (3 * stages);
  const uint32_t tmem_empty = sbase + p.bar_off + 8u * (3 * stages + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (3 * stages + 2));
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* shared_flag = tmem_slot + 2;  // epilogue: CTA-wide decisions
  volatile uint32_t* last_cta = tmem_slot + 3;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const uint64_t timeout = p.timeout_ns;
  const int layers = p.layers;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(full_in(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(accum_full, 1);
    mbar_init(tmem_empty, kChainEpiWarps);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tmem_sf = tmem_base + BM;  // per stage: 8 weight-scale columns, then 8 activation-scale columns

  if (warp == 0) {
    // ------------------------------------------------------------------ weight tiles
    // Weights are read-only for the launch (the same contract as the
    // single-layer kernel), so they load before the wait for the previous grid.
    const bool leader = elect_one();
    const uint64_t policy = policy_evict_first();
    if (!p.weights_early) grid_dependency_wait();
    int t = 0;
    bool stop = false;
    for (int l = 0; l < layers && !stop; ++l) {
      const ChainLayerArgs L = p.layer[l];  // a copy: read once, not through a param-space pointer
      for (int i = b; i < L.items && !stop; i += G) {
        const ChainItem it = chain_item(L, i);
        for (int kt = it.kt0; kt < it.kt1; ++kt, ++t) {
          const int s = t % stages, round = t / stages;
          bool ok = *abort_flag == 0u;
          if (ok && round > 0) ok = mbar_wait(empty(s), (round - 1) & 1, timeout);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            if (leader && *abort_flag == 0u) report_error(p.err, kErrWaitEmpty);
            *abort_flag = 1u;
            stop = true;
            break;
          }
          if (leader) {
            const uint32_t bar = full_w(s);
            mbar_arrive_expect_tx(bar, kTileN * kTileKBytes + kSfTileBytes);
            tma_load_2d(sbase + s * (kTileN * kTileKBytes), &p.wmap[l], kt * kTileKBytes, it.n_tile * kTileN, bar,
                        policy);
            bulk_load(sbase + p.sfw_off + s * kSfTileBytes,
                      L.b_sf + (static_cast<size_t>(it.n_tile) * L.k_tiles + kt) * kSfTileBytes, kSfTileBytes, bar,
                      policy);
          }
          __syncwarp();
        }
      }
    }
    // every copy issued must land before the CTA can exit
    for (int s = 0; s < stages && s < t; ++s) {
      const int last = s + stages * ((t - 1 - s) / stages);
      if (!mbar_wait(full_w(s), (last / stages) & 1, timeout) && leader) report_error(p.err, kErrWaitDrain);
    }
    grid_launch_dependents();
    __syncwarp();
  } else if (warp == kChainActWarp) {
    // ------------------------------------------------------------------ activation tiles
    const uint64_t policy = policy_evict_last();  // codes are shared by every N tile
    grid_dependency_wait();
    int t = 0;
    bool stop = false;
    for (int l = 0; l < layers && !stop; ++l) {
      const ChainLayerArgs L = p.layer[l];  // a copy: read once, not through a param-space pointer
      for (int i = b; i < L.items && !stop; i += G) {
        const ChainItem it = chain_item(L, i);
        for (int kt = it.kt0; kt < it.kt1; ++kt, ++t) {
          const int s = t % stages, round = t / stages;
          bool ok = *abort_flag == 0u;
          if (ok && round > 0) ok = mbar_wait(empty(s), (round - 1) & 1, timeout);
          uint32_t err_bit = kErrWaitEmpty;
          if (lane == 0 && ok) {
            // the activation's K tile: every producer of it has released its counter
            // (each split CTA of a producer tile counts its share of the tile)
            const uint32_t expect = L.in_n_tiles == 0 ? static_cast<uint32_t>(BM / 16)
                                                      : static_cast<uint32_t>(min(2, L.in_n_tiles - 2 * kt) * L.in_splits);
            ok = wait_count_eq(L.in_done + static_cast<size_t>(it.m_tile) * L.k_tiles + kt, expect, timeout);
            err_bit = kErrWaitFlag;
            if (ok) {
              fence_proxy_async_global();  // the TMA reads below come after the acquire
              const uint32_t bar = full_in(s);
              mbar_arrive_expect_tx(bar, p.a_box_rows * kTileKBytes + kChainATileSf);
              tma_load_2d(sbase + p.a_off + s * kATileBytes, &p.amap[l], kt * kTileKBytes, it.m_tile * BM, bar, policy);
              bulk_load(sbase + p.sfa_off + s * kChainATileSf,
                        L.in_sf + (static_cast<size_t>(it.m_tile) * L.k_tiles + kt) * kChainATileSf, kChainATileSf,
                        bar, policy);
            }
          }
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            if (lane == 0 && *abort_flag == 0u) report_error(p.err, err_bit);
            *abort_flag = 1u;
            stop = true;
            break;
          }
        }
      }
    }
    for (int s = 0; s < stages && s < t; ++s) {
      const int last = s + stages * ((t - 1 - s) / stages);
      if (!mbar_wait(full_in(s), (last / stages) & 1, timeout) && lane == 0) report_error(p.err, kErrWaitDrain);
    }
    grid_launch_dependents();
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    int t = 0, item_idx = 0;
    for (int l = 0; l < layers; ++l) {
      const ChainLayerArgs L = p.layer[l];  // a copy: read once, not through a param-space pointer
      const int K = L.K;
      for (int i = b; i < L.items; i += G, ++item_idx) {
        const ChainItem it = chain_item(L, i);
        bool alive = !__any_sync(0xFFFFFFFFu, *abort_flag != 0u);
        if (alive && item_idx > 0) {
          // the epilogue has read the previous item's accumulator
          alive = __all_sync(0xFFFFFFFFu, mbar_wait(tmem_empty, (item_idx - 1) & 1, timeout));
          if (!alive && leader) report_error(p.err, kErrWaitAccum);
        }
        bool first = true;
        for (int kt = it.kt0; kt < it.kt1; ++kt, ++t) {
          const int s = t % stages, round = t / stages;
          if (__any_sync(0xFFFFFFFFu, !alive || *abort_flag != 0u)) {  // warp-uniform
            alive = false;
            continue;
          }
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_w(s), round & 1, timeout))) {
            if (leader) report_error(p.err, kErrWaitTma);
            alive = false;
            continue;
          }
          tc_fence_after_sync();
          const uint32_t sfw_t = tmem_sf + s * 16, sfa_t = sfw_t + 8;
          if (leader) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tmem_cp_32x128b_warpx4(sfw_t + 4 * c,
                                     smem_desc(sbase + p.sfw_off + s * kSfTileBytes + c * kSfChunkBytes, 128, 128, 0));
          }
          __syncwarp();
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_in(s), round & 1, timeout))) {
            if (leader) report_error(p.err, kErrWaitA);
            alive = false;
            continue;
          }
          tc_fence_after_sync();
          if (leader) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tmem_cp_32x128b_warpx4(sfa_t + 4 * c,
                                     smem_desc(sbase + p.sfa_off + s * kChainATileSf + c * kSfChunkBytes, 128, 128, 0));
            const uint64_t a_desc = smem_desc(sbase + s * (kTileN * kTileKBytes), 16, 1024, 2);
            const uint64_t b_desc = smem_desc(sbase + p.a_off + s * kATileBytes, 16, 1024, 2);
            // a whole K tile: four MMAs with compile-time operand offsets and no
            // per-step bound (the issuing lane's instructions set the MMA rate)
            const int steps = kt * kTileK + kTileK <= K ? 4 : (K - kt * kTileK + 63) / 64;
            if (steps == 4) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_mxf4(tmem_base, a_desc + 2 * j, b_desc + 2 * j, mxf4_idesc<BM>((j & 1) * 2), sfw_t + 4 * (j >> 1),
                         sfa_t + 4 * (j >> 1), (first && j == 0) ? 0u : 1u);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if (j >= steps) break;
                const uint32_t sid = (j & 1) * 2;
                mma_mxf4(tmem_base, a_desc + 2 * j, b_desc + 2 * j, mxf4_idesc<BM>(sid), sfw_t + 4 * (j >> 1),
                         sfa_t + 4 * (j >> 1), (first && j == 0) ? 0u : 1u);
              }
            }
            tc_commit(empty(s));  // the stage is free once these MMAs have read it
          }
          first = false;
          __syncwarp();
        }
        if (!alive) *abort_flag = 1u;
        if (leader) tc_commit(accum_full);  // always: the epilogue waits on it once per item
        __syncwarp();
      }
    }
    grid_launch_dependents();
  } else {
    // ------------------------------------------------------------------ activation quantization, epilogues
    const int tid = threadIdx.x - 64;
    const int ew = warp - 2;
    grid_dependency_wait();  // A, C and the workspace may belong to the previous grid
    const int M = p.M;

    // The first layer's activation, quantized once across the grid: unit u is
    // 16 rows x one K tile of 256; CTA G-1-u % G takes it (CTAs past the first
    // layer's items are idle there).  One thread per 16 elements, two lanes per
    // 32-element block (the quantize kernel's scheme).
    {
      const int groups = BM / 16;
      const int units = p.m_tiles * p.k_tiles0 * groups;
      for (int u = G - 1 - b; u < units; u += G) {
        const int g = u % groups, rest = u / groups;
        const int kt = rest % p.k_tiles0, m_tile = rest / p.k_tiles0;
        const int r_t = 16 * g + (tid >> 4), j = tid & 15;
        const int m = m_tile * BM + r_t;
        const int col = kt * kTileK + j * 16;
        const bool valid = m < M && col < p.K0 &&
                           MXFP4_IN_BOUNDS(static_cast<int64_t>(m) * p.lda + col + 16 <= static_cast<int64_t>(M) * p.lda &&
                                               static_cast<int64_t>(m) * (p.K0 / 2) + col / 2 + 8 <=
                                                   static_cast<int64_t>(M) * (p.K0 / 2),
                                           p.err);
        uint4 v = make_uint4(0, 0, 0, 0), w = make_uint4(0, 0, 0, 0);
        if (valid) {
          const uint16_t* src = p.a + static_cast<int64_t>(m) * p.lda + col;
          v = ld_after_wait_v4(src);
          w = ld_after_wait_v4(src + 8);
        }
        uint32_t amax = absmax16_bf16(v, w);
        amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        const uint32_t byte = scale_byte_from_amax(amax);
        const uint16_t sbf = scale_bf16_from_byte(byte);
        const uint32_t c0 = e2m1_pack8(v, sbf), c1 = e2m1_pack8(w, sbf);
        if (valid)
          *reinterpret_cast<uint2*>(p.a_codes + static_cast<int64_t>(m) * (p.K0 / 2) + col / 2) = make_uint2(c0, c1);
        if (m < M && (j & 1) == 0) {
          const int blk = j >> 1;  // blocks past K get scale byte 0 (their codes read as zero)
          p.a_sf[(static_cast<size_t>(m_tile) * p.k_tiles0 + kt) * kChainATileSf + (blk >> 2) * kSfChunkBytes +
                 sf_chunk_offset(r_t) + (blk & 3)] = static_cast<uint8_t>(byte);
        }
        fence_proxy_async_global();  // read by TMA in other CTAs
        named_barrier(1, kChainEpiThreads);  // every thread's stores, then one release add
        if (tid == 0) red_release_gpu_add(p.a_done + static_cast<size_t>(m_tile) * p.k_tiles0 + kt, 1u);
      }
    }

    const int q = warp & 3;  // tensor-memory lane quarter this warp may read: output columns 32q..32q+31
    const int h = ew >> 2;   // which half of the 16-row chunks
    uint16_t* ctile = reinterpret_cast<uint16_t*>(smem + p.epi_off);  // bf16 [BM][128]: this CTA's finished rows
    int item_idx = 0;
    for (int l = 0; l < layers; ++l) {
      const ChainLayerArgs L = p.layer[l];  // a copy: read once, not through a param-space pointer
      const int N = L.N;
      const bool quant_next = L.out_codes != nullptr;
      for (int i = b; i < L.items; i += G, ++item_idx) {
        const ChainItem it = chain_item(L, i);
        const int m_base = it.m_tile * BM;
        const int m_valid = min(BM, M - m_base);
        const int chunks = (m_valid + 15) >> 4;
        const int n_base = it.n_tile * kTileN;
        const bool ok = mbar_wait(accum_full, item_idx & 1, timeout);
        if (!ok) {
          report_error(p.err, kErrWaitAccum);
          *abort_flag = 1u;
        }
        tc_fence_after_sync();
        named_barrier(1, kChainEpiThreads);
        if (tid == 0) *shared_flag = *abort_flag == 0u ? 1u : 0u;
        named_barrier(1, kChainEpiThreads);
        const bool alive = *shared_flag != 0u;

        // One finished value (row m of the tile, column nl), rounded to bf16,
        // into the staged tile.
        auto put = [&](float v, int m, int nl) { ctile[m * kTileN + nl] = __bfloat16_as_ushort(__float2bfloat16_rn(v)); };
        // The staged rows the predicate selects, out: to C (16 bytes at a time
        // where N allows), and, unless this is the last layer, as the next
        // layer's codes and scales -- one thread per 16 elements, two per
        // 32-element block (the quantize kernel's scheme and arithmetic, on the
        // bf16 values of C).  When quantizing, N % 32 == 0, so a block is wholly
        // inside or past N; blocks past N hold zeros (padding weight rows) and
        // get scale byte 0.
        auto write_rows = [&](int units, auto row_of) {
          const int span = (units + 31) / 32 * 32;  // whole warps: the pair shuffle needs every lane
          const bool vec = N % 8 == 0;
          for (int u = tid; u < span; u += kChainEpiThreads) {
            const int m = u < units ? row_of(u >> 3) : 0, j = u & 7;
            const bool valid = u < units && m < m_valid;
            const int n0 = n_base + 16 * j;
            uint4 v = make_uint4(0, 0, 0, 0), w = make_uint4(0, 0, 0, 0);
            if (valid) {
              const uint4* src = reinterpret_cast<const uint4*>(ctile + m * kTileN + 16 * j);
              v = src[0];
              w = src[1];
              uint16_t* crow = reinterpret_cast<uint16_t*>(L.c) + static_cast<int64_t>(m_base + m) * N;
              // (no early exit: every lane reaches the pair shuffle below)
              if (!MXFP4_IN_BOUNDS(m_base + m < M, p.err)) {
              } else if (vec && n0 + 16 <= N) {
                *reinterpret_cast<uint4*>(crow + n0) = v;
                *reinterpret_cast<uint4*>(crow + n0 + 8) = w;
              } else if (vec && n0 + 8 <= N) {
                *reinterpret_cast<uint4*>(crow + n0) = v;
              } else if (n0 < N) {
                const uint16_t* e16 = ctile + m * kTileN + 16 * j;
                for (int e = 0; e < 16 && n0 + e < N; ++e) crow[n0 + e] = e16[e];
              }
            }
            if (!quant_next) continue;  // uniform
            uint32_t amax = absmax16_bf16(v, w);
            amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            const uint32_t byte = scale_byte_from_amax(amax);
            const uint16_t sbf = scale_bf16_from_byte(byte);
            const uint32_t c0 = e2m1_pack8(v, sbf), c1 = e2m1_pack8(w, sbf);
            if (valid && n_base + 16 * j < N &&
                MXFP4_IN_BOUNDS(static_cast<int64_t>(m_base + m) * (N / 2) + n_base / 2 + 8 * j + 8 <=
                                    static_cast<int64_t>(M) * (N / 2),
                                p.err))
              *reinterpret_cast<uint2*>(L.out_codes + static_cast<int64_t>(m_base + m) * (N / 2) + n_base / 2 + 8 * j) =
                  make_uint2(c0, c1);
            if (valid && (j & 1) == 0)
              L.out_sf[(static_cast<size_t>(it.m_tile) * L.k_tiles_next + (it.n_tile >> 1)) * kChainATileSf +
                       (it.n_tile & 1) * kSfChunkBytes + sf_chunk_offset(m) + (j >> 1)] = static_cast<uint8_t>(byte);
          }
        };
        // Counts this CTA's part of the tile done.  The CTA barrier orders every
        // thread's stores before the single release add (release is cumulative).
        auto release = [&]() {
          fence_proxy_async_global();  // codes and scales are read by TMA in other CTAs
          named_barrier(1, kChainEpiThreads);
          if (tid == 0 && alive && L.out_done != nullptr)
            red_release_gpu_add(L.out_done + static_cast<size_t>(it.m_tile) * L.k_tiles_next + (it.n_tile >> 1), 1u);
        };

        if (L.splits == 1) {
#pragma unroll 1
          for (int c = h; c < chunks; c += 2) {
            if (!alive) break;
            uint32_t r[16];
            tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (16 * c + e < m_valid) put(__uint_as_float(r[e]), 16 * c + e, 32 * q + lane);
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(tmem_empty);
          named_barrier(1, kChainEpiThreads);  // the staged tile is complete
          if (alive) write_rows(m_valid * 8, [](int row) { return row; });
          release();
        } else {
          // K split: every split stores its fp32 partial; once all S have
          // (a count per tile), split CTA s finishes the tile's 4-row groups
          // g = s, s + S, ..., each value the sum of the S partials in split
          // order (deterministic: the same order whichever CTA sums).
          const int S = L.splits;
          const int tile = it.m_tile * L.n_tiles + it.n_tile;
          float* part = L.partials + static_cast<size_t>(tile) * S * BM * kTileN;
#pragma unroll 1
          for (int c = h; c < chunks; c += 2) {
            if (!alive) break;
            uint32_t r[16];
            tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 16, r);
            tmem_ld_wait();
            float* dst = part + (static_cast<size_t>(it.split) * BM + 16 * c) * kTileN + 32 * q + lane;
            if (!MXFP4_IN_BOUNDS(tile < L.n_tiles * p.m_tiles && it.split < S, p.err)) break;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (16 * c + e < m_valid) dst[e * kTileN] = __uint_as_float(r[e]);
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(tmem_empty);
          named_barrier(1, kChainEpiThreads);
          if (tid == 0) {
            bool all = false;
            if (alive) {
              red_release_gpu_add(L.tickets + tile, 1u);
              all = wait_count_eq(L.tickets + tile, static_cast<uint32_t>(S), timeout);
              if (!all) {
                report_error(p.err, kErrWaitFlag);
                *abort_flag = 1u;
              }
            }
            *shared_flag = all ? 1u : 0u;
          }
          named_barrier(1, kChainEpiThreads);
          const bool summing = *shared_flag != 0u;
          const int groups = (m_valid + 3) >> 2;
          const int mine = summing && it.split < groups ? (groups - it.split + S - 1) / S : 0;
          // 16 pieces (row, 32 columns) per group, piece p of the CTA's groups
          // taken by warp p % 8; each lane loads the S partials of its column
          // for as many pieces as fit 16 values in flight, then sums each in
          // split order
          const int pieces = mine * 16;
          auto reduce = [&](auto splits) {
            constexpr int SS = decltype(splits)::value;
            constexpr int B = 2 * kMaxSplits / SS;  // pieces per round: 16 values in flight
#pragma unroll 1
            for (int p0 = ew; p0 < pieces; p0 += kChainEpiWarps * B) {
              float v[B][SS];
#pragma unroll
              for (int bp = 0; bp < B; ++bp) {
                const int piece = p0 + kChainEpiWarps * bp;
                const int g = it.split + SS * (piece >> 4), row = 4 * g + ((piece & 15) >> 2), qq = piece & 3;
                const bool in = piece < pieces && row < m_valid;
#pragma unroll
                for (int s2 = 0; s2 < SS; ++s2)
                  v[bp][s2] = in ? __ldcg(part + (static_cast<size_t>(s2) * BM + row) * kTileN + 32 * qq + lane) : 0.0f;
              }
#pragma unroll
              for (int bp = 0; bp < B; ++bp) {
                const int piece = p0 + kChainEpiWarps * bp;
                const int g = it.split + SS * (piece >> 4), row = 4 * g + ((piece & 15) >> 2), qq = piece & 3;
                float f = v[bp][0];
#pragma unroll
                for (int s2 = 1; s2 < SS; ++s2) f += v[bp][s2];
                if (piece < pieces && row < m_valid) put(f, row, 32 * qq + lane);
              }
            }
          };
          switch (S) {
            case 2: reduce(std::integral_constant<int, 2>{}); break;
            case 3: reduce(std::integral_constant<int, 3>{}); break;
            case 4: reduce(std::integral_constant<int, 4>{}); break;
            case 5: reduce(std::integral_constant<int, 5>{}); break;
            case 6: reduce(std::integral_constant<int, 6>{}); break;
            case 7: reduce(std::integral_constant<int, 7>{}); break;
            default: reduce(std::integral_constant<int, 8>{}); break;
          }
          named_barrier(1, kChainEpiThreads);  // the staged rows are complete
          if (mine > 0) write_rows(mine * 32, [&](int r) { return 4 * (it.split + S * (r >> 2)) + (r & 3); });
          release();
        }
      }
    }
    grid_launch_dependents();
  }

  // ---------------------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
  // The last CTA to get here clears every counter for the next launch (all
  // other CTAs are past their last wait).  Only threads that waited for the
  // previous grid touch the workspace.
  if (threadIdx.x == 64) {
    __threadfence();
    *last_cta = atom_add_acq_rel_gpu(p.exit_count, 1u) == static_cast<uint32_t>(G - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (*last_cta != 0u && warp >= 2 && warp < kChainActWarp) {
    for (int i = threadIdx.x - 64; i < p.n_counters; i += kChainEpiThreads) p.counters[i] = 0u;
  }
}

template <int BM>
static cudaError_t launch_chain_t(const ChainArgs& args, int grid, int smem_bytes, bool programmatic,
                                  cudaStream_t s) {
  auto kernel = chain_kernel<BM>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kChainThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

cudaError_t launch_chain(const ChainArgs& args, int block_m, int grid, int smem_bytes, bool programmatic,
                         cudaStream_t s) {
  switch (block_m) {
    case 16: return launch_chain_t<16>(args, grid, smem_bytes, programmatic, s);
    case 32: return launch_chain_t<32>(args, grid, smem_bytes, programmatic, s);
    case 64: return launch_chain_t<64>(args, grid, smem_bytes, programmatic, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int BM>
static int blocks_per_sm_t(int smem_bytes) {
  auto kernel = chain_kernel<BM>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kChainThreads, static_cast<size_t>(smem_bytes)) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int chain_blocks_per_sm(int block_m, int smem_bytes) {
  switch (block_m) {
    case 16: return blocks_per_sm_t<16>(smem_bytes);
    case 32: return blocks_per_sm_t<32>(smem_bytes);
    case 64: return blocks_per_sm_t<64>(smem_bytes);
    default: return 0;
  }
}

}  // namespace mxfp4
