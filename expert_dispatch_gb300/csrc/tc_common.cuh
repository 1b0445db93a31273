// tc_common.cuh -- pieces shared by the tcgen05 grouped GEMMs (bf16 weights in
// tc_gemm.cu, Q8_0 weights in tc_gemm_q8.cu): work-unit schedule, bounded
// waits, the TMEM epilogue, and tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace tc {

constexpr int MODE_ROUTER = 0, MODE_GATEUP = 1, MODE_DOWN = 2;
constexpr int kMaxGroups = 1028;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter

struct Params {
  const int32_t* offsets;  // [n_groups + 1] batch boundaries, or null
  int n_groups;
  int rows_single;         // rows of the single group when offsets is null
  int Mg;                  // weight rows per group
  int K;                   // reduction length (multiple of 64)
  void* out;
  int ldo;                 // output row stride, elements
  const float* row_scale;  // MODE_DOWN: per-row factor or null
  int* err;
  int max_rows;            // rows of the token operand / output; batch bounds are clamped to it
  int ksplit;              // MODE_ROUTER: K is cut into ksplit chunks of kb_per 64-wide blocks,
  int kb_per;              //   each chunk's partial sums go to out + chunk * rows * ldo
  const int32_t* group_slot;  // [n_groups] weight matrix of each group (null: group g uses
                              //   matrix g); a negative entry skips the group
};

// The weight matrix group g reads: its slot in a slot pool, or g itself.
__device__ __forceinline__ int weight_mat(const Params& p, int g) {
  return p.group_slot ? p.group_slot[g] : g;
}

struct Unit {
  int g, mt, r0, nt, kb0, kb1;
};

// Unit u -> (group, weight block, token rows, K range).  A group with at most
// four token tiles is ordered token-tile-minor (a weight block's tiles run
// back to back, so its bytes come from HBM once); a group with more is
// ordered weight-block-minor (the CTAs running together cover all weight
// blocks of a few token tiles, so the expert's weights and those token rows
// stay in L2 while its tiles are swept).  The router always uses the latter.
template <int MODE, int BN>
__device__ __forceinline__ Unit decode_unit(int u, const int* prefix, const int* gstart,
                                            int n_groups, int m_tiles, int KB, const Params& p) {
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  const int local = u - prefix[lo];
  const int cnt = gstart[lo + 1] - gstart[lo];
  const int tiles = (cnt + BN - 1) / BN;
  int mt, tt, ks = 0;
  if (MODE == MODE_ROUTER) {
    mt = local % m_tiles;
    const int rest = local / m_tiles;
    tt = rest % tiles;
    ks = rest / tiles;
  } else if (tiles <= 4) {  // few token tiles: a weight block's tiles back to back
    mt = local / tiles;
    tt = local - mt * tiles;
  } else {  // many token tiles: all weight blocks of a token tile back to back
    mt = local % m_tiles;
    tt = local / m_tiles;
  }
  Unit r;
  r.g = lo;
  r.mt = mt;
  r.r0 = gstart[lo] + tt * BN;
  r.nt = min(BN, cnt - tt * BN);
  r.kb0 = MODE == MODE_ROUTER ? ks * p.kb_per : 0;
  r.kb1 = MODE == MODE_ROUTER ? min(KB, r.kb0 + p.kb_per) : KB;
  return r;
}

// SM pairs: MMA width of a unit with nt token rows, a multiple of 32 so each
// CTA holds a multiple of 16 rows, brought by one box of that height.
__device__ __forceinline__ int pair_n(int nt) { return max(32, (nt + 31) & ~31); }

// One warp builds the schedule in shared memory.  Batch boundaries are made
// safe first: each clamped to [0, max_rows] and forced non-decreasing
// (running max), so every batch lies inside the row buffers whatever the
// caller passed; any change is flagged.  Then prefix[g] = units before group
// g, with m_tiles x ceil(rows / BN) (x ksplit for the router) units per group;
// a group whose group_slot entry is negative gets none.
template <int MODE, int BN>
__device__ __forceinline__ void build_schedule(const Params& p, int m_tiles, int* prefix,
                                               int* gstart) {
  const int lane = threadIdx.x & 31;
  int run = 0;
  for (int base = 0; base <= p.n_groups; base += 32) {
    const int i = base + lane;
    int v = 0, raw = 0;
    if (i <= p.n_groups) {
      raw = p.offsets ? p.offsets[i] : (i == 0 ? 0 : p.rows_single);
      v = min(max(raw, 0), p.max_rows);
    }
    int m = max(v, run);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) m = max(m, __shfl_up_sync(0xffffffffu, m, o));
    if (i <= p.n_groups) {
      gstart[i] = m;
      if (m != raw) flag_error(p.err, kErrDeviceInput);
    }
    run = __shfl_sync(0xffffffffu, m, 31);
  }
  __syncwarp();
  int carry = 0;
  if (lane == 0) prefix[0] = 0;
  for (int base = 0; base < p.n_groups; base += 32) {
    const int g = base + lane;
    int units = 0;
    if (g < p.n_groups && !(p.group_slot && p.group_slot[g] < 0)) {
      const int cnt = gstart[g + 1] - gstart[g];
      units = m_tiles * ((cnt + BN - 1) / BN) * (MODE == MODE_ROUTER ? p.ksplit : 1);
    }
    int incl = units;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (g < p.n_groups) prefix[g + 1] = carry + incl;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Warp-uniform bounded wait: every lane polls, the timeout decision is lane 0's.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* err) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;  // the common case
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((i & 31u) == 31u) {
      int stop = 0;
      if ((threadIdx.x & 31) == 0) {
        if (*abort_flag) {
          stop = 1;
        } else if (globaltimer_ns() - t0 > kWaitLimitNs) {
          *abort_flag = 1;
          flag_error(err, kErrTimeout);
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

// Bounded wait used while winding down: ignores the abort flag.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity, int* err) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      flag_error(err, kErrTimeout);
      return;
    }
  }
}

// Epilogue, run by the kEpiWarps epilogue warps (warp indices first_warp ..
// first_warp + 7): for every unit of this CTA, wait for its accumulators in
// TMEM, read them with tcgen05.ld (a warp may only read its lane quarter,
// warp % 4; the two warps of a quarter take alternate 16-column chunks) and
// apply the mode's epilogue.
//   MODE_ROUTER : partial logits, fp32, stored straight from the loads
//   MODE_GATEUP : H = silu(gate) * up, bf16 (fp16 when H_F16; a value beyond
//                 fp16's range is flagged as an input error); silu_fast
//   MODE_DOWN   : y_perm = acc * row_scale, bf16 (whatever H_F16)
// For the last two the whole unit is first turned into packed 16-bit pairs
// held in registers; the TMEM buffer is handed back before the global
// stores, so those overlap the next unit's MMAs instead of delaying them.
// With NPART > 1 the unit's K blocks were accumulated into NPART partial
// sets (K block j of the unit into set j % NPART, NACC * BN columns apart),
// added here in set order; a unit with fewer K blocks than sets has only
// the first ones.
//
// Units u0, u0 + ustride, ... are this CTA's; a unit's weight block covers
// rows mt * MT + row_off .. + 127 of the group, or, for MODE_DOWN with two
// accumulators (MT = 256 on one SM), rows mt * 256 .. + 255: the first
// accumulator holds the upper 128, the second the lower.  With PAIR the accumulator
// buffers are released on the even CTA of the cluster (the pair's MMA
// issuer), whatever CTA this is.
template <int MODE, int BN, int NACC, int NBUF, bool H_F16 = false, int NPART = 1, int MT = 128,
          bool PAIR = false>
__device__ __forceinline__ void epilogue_loop(const Params& p, int total, int m_tiles, int KB,
                                              const int* prefix, const int* gstart,
                                              uint32_t tmem_base, uint32_t accf0,
                                              uint32_t acce0, volatile int* abort_flag,
                                              int first_warp, int u0, int ustride, int row_off) {
  constexpr int NCH = BN / 32;  // 16-column chunks per thread
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;                   // TMEM lane quarter this warp may access
  const int half = (warp - first_warp) / 4;  // alternate 16-column chunks
  auto release = [&](int buf) {  // lane 0: the accumulator buffer may be overwritten
    if (PAIR)
      mbar_arrive_cluster(mapa_shared(acce0 + 8u * buf, 0));
    else
      mbar_arrive(acce0 + 8u * buf);
  };
  int it = 0;
  for (int u = u0; u < total; u += ustride, ++it) {
    const Unit t = decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
    const int buf = NBUF == 2 ? (it & 1) : 0;
    const uint32_t use = NBUF == 2 ? (uint32_t)(it >> 1) : (uint32_t)it;
    if (!mbar_wait_warp(accf0 + 8u * buf, use & 1u, abort_flag, p.err)) break;
    tc_fence_after();
    const int m = t.mt * MT + row_off + q * 32 + lane;  // weight row within the group
    const bool mvalid = m < p.Mg;
    const uint32_t tb =
        tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * NPART * NACC * BN);
    const int nparts = NPART == 1 ? 1 : min(NPART, t.kb1 - t.kb0);
    // accumulator columns c0 .. c0 + 15 (both operands, partial sets added)
    auto load16 = [&](int c0, uint32_t (&a)[16], uint32_t (&b)[16]) {
      tmem_ld16(tb + c0, a);
      if (NACC == 2) tmem_ld16(tb + BN + c0, b);
      for (int pp = 1; pp < nparts; ++pp) {
        uint32_t a2[16], b2[16];
        const uint32_t tp = tb + (uint32_t)(pp * NACC * BN);
        tmem_ld16(tp + c0, a2);
        if (NACC == 2) tmem_ld16(tp + BN + c0, b2);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          a[j] = __float_as_uint(__uint_as_float(a[j]) + __uint_as_float(a2[j]));
          if (NACC == 2) b[j] = __float_as_uint(__uint_as_float(b[j]) + __uint_as_float(b2[j]));
        }
      }
      tmem_ld_wait();
    };
    if constexpr (MODE == MODE_ROUTER) {
      for (int c0 = 16 * half; c0 < t.nt; c0 += 32) {
        uint32_t a[16], b[16];
        load16(c0, a, b);
        if (!mvalid) continue;
        const size_t chunk = (size_t)(t.kb0 / p.kb_per);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = c0 + j;
          if (col >= t.nt) break;
          const size_t row = (size_t)(t.r0 + col);
          static_cast<float*>(p.out)[(chunk * p.rows_single + row) * p.ldo + m] =
              __uint_as_float(a[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(buf);
    } else if constexpr (MODE == MODE_DOWN && NACC == 2) {
      // Two stacked 128-row weight blocks (a unit of MT = 256 rows): warps
      // 0-3 of the epilogue take the first accumulator, 4-7 the second, each
      // over all of the tile's columns.
      static_assert(NPART == 1 && !PAIR && MT == 256, "stacked down accumulators");
      constexpr int NC2 = BN / 16;
      const int m2 = t.mt * MT + row_off + half * 128 + q * 32 + lane;
      const uint32_t ta = tb + (uint32_t)(half * BN);
      uint32_t a[NC2][16];
#pragma unroll
      for (int i = 0; i < NC2; ++i)
        if (16 * i < t.nt) tmem_ld16(ta + 16 * i, a[i]);  // warp-uniform
      tmem_ld_wait();
      uint32_t pk[NC2][8];
#pragma unroll
      for (int i = 0; i < NC2; ++i) {
        const int c0 = 16 * i;
        if (c0 >= t.nt) break;  // warp-uniform: the chunks that were loaded
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float v0 = __uint_as_float(a[i][j]), v1 = __uint_as_float(a[i][j + 1]);
          if (p.row_scale) {  // read for batch rows only
            if (c0 + j < t.nt) v0 *= p.row_scale[t.r0 + c0 + j];
            if (c0 + j + 1 < t.nt) v1 *= p.row_scale[t.r0 + c0 + j + 1];
          }
          const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
          pk[i][j / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(buf);  // TMEM free: stores follow
      if (m2 < p.Mg) {
        uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
        for (int i = 0; i < NC2; ++i) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = 16 * i + j;
            if (col >= t.nt) break;
            const uint32_t w = pk[i][j / 2];
            out[(size_t)(t.r0 + col) * p.ldo + m2] =
                (uint16_t)((j & 1) ? (w >> 16) : (w & 0xffffu));
          }
        }
      }
    } else {
      uint32_t pk[NCH][8];  // the unit's results, packed 16-bit pairs
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int c0 = 16 * half + 32 * i;
        if (c0 >= t.nt) break;  // warp-uniform
        uint32_t a[16], b[16];
        load16(c0, a, b);
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float v0 = __uint_as_float(a[j]), v1 = __uint_as_float(a[j + 1]);
          if (MODE == MODE_GATEUP) {
            v0 = silu_fast(v0) * __uint_as_float(b[j]);
            v1 = silu_fast(v1) * __uint_as_float(b[j + 1]);
          } else if (p.row_scale) {
            const int col = c0 + j;  // row_scale is read for batch rows only
            if (col < t.nt) v0 *= p.row_scale[t.r0 + col];
            if (col + 1 < t.nt) v1 *= p.row_scale[t.r0 + col + 1];
          }
          if (H_F16 && MODE == MODE_GATEUP) {
            const __half2 h = __floats2half2_rn(v0, v1);
            const bool inf0 = c0 + j < t.nt && __hisinf(__low2half(h));
            const bool inf1 = c0 + j + 1 < t.nt && __hisinf(__high2half(h));
            if (mvalid && (inf0 || inf1)) flag_error(p.err, kErrDeviceInput);
            pk[i][j / 2] = *reinterpret_cast<const uint32_t*>(&h);
          } else {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
            pk[i][j / 2] = *reinterpret_cast<const uint32_t*>(&h);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(buf);  // TMEM free: stores follow
      if (mvalid) {
        uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          const int c0 = 16 * half + 32 * i;
          if (c0 >= t.nt) break;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col >= t.nt) break;
            const uint32_t w = pk[i][j / 2];
            out[(size_t)(t.r0 + col) * p.ldo + m] =
                (uint16_t)((j & 1) ? (w >> 16) : (w & 0xffffu));
          }
        }
      }
    }
  }
}

}  // namespace tc

// Token-row maps of one operand for the SM-pair GEMMs: box[i] is (i + 1) * 16
// rows high (up to 128, half of the largest tile), so each CTA brings its
// share of a tile's token rows with one copy per K block.
struct PairTokenMaps {
  CUtensorMap box[8];
};

// The FFN's GEMMs on SM pairs (tc_gemm_pair.cu), weight maps with 128-row
// boxes: gate/up with 160-row token tiles (token maps of x_perm, box[0..4]),
// down with 256-row tiles (token maps of H, box[0..7]).
cudaError_t launch_gateup_pair(const CUtensorMap& tg, const CUtensorMap& tu,
                               const PairTokenMaps& tx, const tc::Params& p, int P, int n_groups,
                               cudaStream_t s);
cudaError_t launch_down_pair(const CUtensorMap& td, const PairTokenMaps& th, const tc::Params& p,
                             int P, int n_groups, cudaStream_t s);

// Host: 2-D tiled tensor map (row-major [rows, inner] of `elsize`-byte elements),
// boxes of box_rows x box_inner, with the given shared-memory swizzle (the MMA
// operands use 128-byte swizzle with 128-byte box rows).
bool make_tmap_2d(CUtensorMap* tm, const void* base, CUtensorMapDataType dtype, int elsize,
                  uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                  CUtensorMapSwizzle swizzle);

}  // namespace moe
