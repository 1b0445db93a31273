// tc_gemm_pair.cu -- the expert FFN's grouped GEMMs for large token tiles, run
// on pairs of SMs ("Distributed MoE" (tenzro docs), expert FFN: each expert
// applies its SwiGLU projections, Y = X * W^T, to the batch of tokens routed
// to it).
//
// Same batches, schedule order and epilogue as the one-SM kernel (tc_gemm.cu);
// what changes is the tile.  A unit here is (group, 256 weight rows, up to BN
// token rows, all of K), and a cluster of two CTAs on two SMs runs it as one
// M = 256 tcgen05 tile (cta_group::2):
//   * CTA r loads weight rows 128 r .. 128 r + 127 of the block and half of the
//     token rows (N / 2 rows from r0 + r N / 2) into its own shared memory; both
//     CTAs' copies complete on the even CTA's stage barrier;
//   * one thread of the even CTA issues the MMAs, which read both CTAs'
//     operands, and commits each stage's release and each unit's accumulators
//     to the barriers of both CTAs (multicast);
//   * each CTA's epilogue reads its own 128 accumulator lanes and releases the
//     buffer on the even CTA's barrier (which counts both CTAs' warps).
// Per SM and K block this moves half the token bytes of the one-SM kernel for
// the same MMA work, so the shared-memory stages go further and the L2 feed
// per flop drops; it is used where token tiles are large (prefill-sized
// batches), where that feed, not HBM, bounds the one-SM kernel.
//
// Every wait is bounded (tc_common.cuh); a CTA that gives up raises its abort
// flag, and its partner's waits then expire in turn.  Both CTAs meet at a
// cluster barrier before the pair's TMEM is freed, after the even CTA has
// waited for every MMA it issued and every stage it armed.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {
namespace {

using tc::MODE_DOWN;
using tc::MODE_GATEUP;
using tc::Params;
using tc::pair_n;
using tc::Unit;
constexpr int kThreads = 32 * (2 + tc::kEpiWarps);  // producer, MMA, epilogue

template <int MODE, int BN, int STAGES>
struct CfgPair {
  static constexpr int NA = MODE == MODE_GATEUP ? 2 : 1;  // weight operands per stage
  static constexpr int A_BYTES = 128 * 64 * 2;            // this CTA's 128 weight rows
  static constexpr int B_BYTES = (BN / 2) * 128;          // this CTA's half of the tokens
  static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
  static constexpr int NACC = NA;
  static constexpr int NBUF = 2 * NACC * BN <= 512 ? 2 : 1;
  static constexpr int COLS = NBUF * NACC * BN;
  static constexpr int TMEM_COLS =
      COLS <= 32 ? 32 : COLS <= 64 ? 64 : COLS <= 128 ? 128 : COLS <= 256 ? 256 : 512;
  static constexpr int NBARS = 2 * STAGES + 2 * NBUF + 1;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int PREFIX_OFF = MISC_OFF + 16;
  static constexpr int GSTART_OFF = PREFIX_OFF + 4 * (tc::kMaxGroups + 1);
  static constexpr int SMEM_TOTAL = GSTART_OFF + 4 * (tc::kMaxGroups + 1) + 1024;
  static_assert(BN % 64 == 0 || BN == 160, "token tile: halves of whole 16-row boxes");
  static_assert(BN >= 64 && BN <= 256, "token tile");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(COLS <= 512, "TMEM columns");
  static_assert(SMEM_TOTAL <= 232448, "shared memory");
};

template <int MODE, int BN, int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA0,
                         const __grid_constant__ CUtensorMap tmA1,
                         const __grid_constant__ PairTokenMaps tmB, const Params p) {
  using C = CfgPair<MODE, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t accf0 = bar0 + 8u * (2 * STAGES);
  const uint32_t acce0 = bar0 + 8u * (2 * STAGES + C::NBUF);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * C::NBUF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  int* prefix = reinterpret_cast<int*>(smem + C::PREFIX_OFF);
  int* gstart = reinterpret_cast<int*>(smem + C::GSTART_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = (int)(blockIdx.x >> 1), n_pairs = (int)(gridDim.x >> 1);
  const int m_tiles = (p.Mg + 255) / 256;
  const int KB = p.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(accf0 + 8u * b, 1);
      mbar_init(acce0 + 8u * b, 2 * tc::kEpiWarps);  // the epilogue warps of both CTAs
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA0);
    if (C::NA == 2) tma_prefetch_desc(&tmA1);
    for (int i = 0; i < BN / 32; ++i) tma_prefetch_desc(&tmB.box[i]);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 2) tc::build_schedule<MODE, BN>(p, m_tiles, prefix, gstart);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = prefix[p.n_groups];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      // bytes one CTA brings per K block of unit t; the even CTA expects both CTAs'
      auto cta_bytes = [&](const Unit& t) {
        return (uint32_t)(C::NA * C::A_BYTES + (pair_n(t.nt) / 2) * 128);
      };
      auto weight_row = [&](const Unit& t) {
        return tc::weight_mat(p, t.g) * p.Mg + t.mt * 256 + (int)rank * 128;
      };
      // The first unit's weight tiles are requested before waiting for the
      // predecessor grid (weights are never written by the kernel just
      // before; the token rows are, and the unit schedule comes from a grid
      // two launches back).
      int n_pre = 0;
      if (pair < total) {
        const Unit t = tc::decode_unit<MODE, BN>(pair, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int arow = weight_row(t);
        n_pre = min(STAGES, t.kb1 - t.kb0);
        for (int i = 0; i < n_pre; ++i) {  // fresh ring: stages 0..n_pre-1 are free
          if (rank == 0) {
            mbar_arrive_expect_tx(full_bar(i), 2 * cta_bytes(t));
            armed |= 1u << i;
          }
          const uint32_t fb = mapa_shared(full_bar(i), 0);
          const uint32_t sA = sbase + i * C::STAGE_BYTES;
          tma_load_2d_pair(sA, &tmA0, fb, (t.kb0 + i) * 64, arow);
          if (C::NA == 2) tma_load_2d_pair(sA + C::A_BYTES, &tmA1, fb, (t.kb0 + i) * 64, arow);
        }
      }
      pdl_wait();
      bool first = true;
      for (int u = pair; u < total && !*abort_flag; u += n_pairs) {
        if (u + n_pairs >= total) pdl_trigger();  // this pair's last unit
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int hb = pair_n(t.nt) / 2;  // token rows this CTA holds
        const int brow = t.r0 + (int)rank * hb;
        const uint32_t bytes = cta_bytes(t);
        const int arow = weight_row(t);
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          const bool pre = first && kb - t.kb0 < n_pre;  // armed, weights already requested
          if (!pre) {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
              ok = false;
              break;
            }
            if (rank == 0) {
              mbar_arrive_expect_tx(full_bar(stage), 2 * bytes);
              armed |= 1u << stage;
              armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            }
          }
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t sA = sbase + stage * C::STAGE_BYTES;
          if (!pre) {
            tma_load_2d_pair(sA, &tmA0, fb, kb * 64, arow);
            if (C::NA == 2) tma_load_2d_pair(sA + C::A_BYTES, &tmA1, fb, kb * 64, arow);
          }
          // this CTA's token rows: one box hb rows high
          tma_load_2d_pair(sA + C::NA * C::A_BYTES, &tmB.box[hb / 16 - 1], fb, kb * 64, brow);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        first = false;
        if (!ok) break;
      }
      if (pair >= total) pdl_trigger();
      if (rank == 0) {
        // wind down: every stage armed here has received both CTAs' copies
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) tc::mbar_wait_drain(full_bar(s), (armed_parity >> s) & 1u, p.err);
      } else if (*abort_flag) {
        // this CTA's copies complete on its partner's barriers: after giving
        // up, leave them a bounded time to land before the shared memory goes
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool issued = false;
      for (int u = pair; u < total && !*abort_flag; u += n_pairs, ++it) {
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const uint32_t idesc = idesc_bf16_f32(256, pair_n(t.nt));
        const int buf = C::NBUF == 2 ? (it & 1) : 0;
        const uint32_t use = C::NBUF == 2 ? (uint32_t)(it >> 1) : (uint32_t)it;
        if (!mbar_wait(acce0 + 8u * buf, (use & 1u) ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(buf * C::NACC * BN);
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sbase + stage * C::STAGE_BYTES;
          const uint32_t sB = sA + C::NA * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(sB + kk * 32);
            const uint32_t acc = (kb != t.kb0 || kk != 0) ? 1u : 0u;
            umma_bf16_pair(d0, smem_desc_sw128(sA + kk * 32), bdesc, idesc, acc);
            if (C::NA == 2)
              umma_bf16_pair(d0 + BN, smem_desc_sw128(sA + C::A_BYTES + kk * 32), bdesc, idesc,
                             acc);
          }
          issued = true;
          umma_commit_pair_mc(empty_bar(stage), 3);  // both CTAs' stage is free again
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(accf0 + 8u * buf, 3);  // both CTAs' accumulators are ready
      }
      // wind down: every MMA issued here has completed before the pair's TMEM is freed
      if (issued) {
        umma_commit_pair_mc(drain_bar, 1);
        tc::mbar_wait_drain(drain_bar, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9, both CTAs)
    tc::epilogue_loop<MODE, BN, C::NACC, C::NBUF, false, 1, 256, true>(
        p, total, m_tiles, KB, prefix, gstart, tmem_base, accf0, acce0, abort_flag, 2, pair,
        n_pairs, (int)rank * 128);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the partner is done with this CTA's shared memory and TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <int MODE, int BN, int STAGES>
cudaError_t launch_pair(const CUtensorMap& a0, const CUtensorMap& a1, const PairTokenMaps& b,
                        const Params& p, long long max_units, const char* name, cudaStream_t s) {
  using C = CfgPair<MODE, BN, STAGES>;
  auto kern = tc_grouped_gemm_pair<MODE, BN, STAGES>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  // clusters that fit on the device at once (an SM pair must share a GPC, so
  // this can be fewer than half the SMs); the grid never exceeds it, so every
  // pair runs its share of the units concurrently
  static int max_clusters[64] = {};
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (max_clusters[dev] == 0) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (unsigned)(num_sms() / 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = C::SMEM_TOTAL;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorInvalidConfiguration;
      max_clusters[dev] = n;
    }
  }
  const long long pairs = max_units < max_clusters[dev] ? max_units : max_clusters[dev];
  if (pairs <= 0) return cudaSuccess;
  ProfScope pr(name, s);
  (void)launch_kernel(kern, (unsigned)(2 * pairs), kThreads, C::SMEM_TOTAL, s, a0, a1, b, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gateup_pair(const CUtensorMap& tg, const CUtensorMap& tu,
                               const PairTokenMaps& tx, const tc::Params& p, int P, int n_groups,
                               cudaStream_t s) {
  const long long units = (long long)((p.Mg + 255) / 256) * ((P + 159) / 160 + n_groups);
  return launch_pair<MODE_GATEUP, 160, 5>(tg, tu, tx, p, units, "ffn_gateup_tc", s);
}

cudaError_t launch_down_pair(const CUtensorMap& td, const PairTokenMaps& th, const tc::Params& p,
                             int P, int n_groups, cudaStream_t s) {
  const long long units = (long long)((p.Mg + 255) / 256) * ((P + 255) / 256 + n_groups);
  return launch_pair<MODE_DOWN, 256, 6>(td, td, th, p, units, "ffn_down_tc", s);
}

}  // namespace moe
