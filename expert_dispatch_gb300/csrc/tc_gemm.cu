// tc_gemm.cu -- grouped GEMM on the 5th-generation tensor cores (tcgen05)
// for the expert FFN and the router of bf16 layers.
//
// What it computes ("Distributed MoE" (tenzro docs), expert-host-runtime and
// compute-seam paragraphs: SwiGLU experts, every projection Y = X * W^T with
// W stored [out, in]; "Expert-sharding" (kvasir wiki), section "Twee rollen":
// the worker's three mat-muls over the rows it was sent):
//   MODE_GATEUP : H[r, n] = silu(X[r] . Wg_e[n]) * (X[r] . Wu_e[n])
//   MODE_DOWN   : Y[r, m] = (H[r] . Wd_e[m]) * row_scale[r]
//   MODE_ROUTER : L[t, e] = x[t] . Wr[e]
// for every batch row r of expert e (rows offsets[e] .. offsets[e+1]).
//
// Design (sm_103a, one CTA per SM, persistent):
//   * Roles are swapped relative to the usual token-major GEMM: the MMA's M
//     side (128 lanes of TMEM) holds 128 weight rows and its N side holds up
//     to BN token rows of the expert's batch, so a batch of any size down to
//     one token costs N = 16 columns instead of a 128-row tile; weights are
//     streamed exactly once per (expert, 128-row block, token tile).
//   * Work unit = (expert, 128-row weight block, token tile).  Units of one
//     weight block are adjacent in the schedule so CTAs running at the same
//     time share its bytes through L2.
//   * Warp 0 lane 0 issues TMA loads (128-byte swizzle) into a STAGES-deep
//     shared-memory ring; warp 1 lane 0 issues tcgen05.mma (bf16 x bf16 ->
//     fp32 in TMEM) and commits each stage back to the loader; warps 2-5 read
//     the accumulators with tcgen05.ld and apply the epilogue (SwiGLU, row
//     scale) while the next unit's MMAs run into the other TMEM buffer.
//   * Token rows are loaded in 32-row boxes, only as many as the unit has.
//   * Every wait is bounded (1 s); on expiry the CTA records a timeout in the
//     error word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int MODE_ROUTER = 0, MODE_GATEUP = 1, MODE_DOWN = 2;
constexpr int kMaxGroups = 1028;
constexpr int kEpiWarps = 8;                   // two per TMEM lane quarter
constexpr int kThreads = 32 * (2 + kEpiWarps);  // producer, MMA, epilogue

template <int MODE, int BN, int STAGES>
struct Cfg {
  static constexpr int NA = MODE == MODE_GATEUP ? 2 : 1;  // weight operands per stage
  static constexpr int A_BYTES = 128 * 64 * 2;
  static constexpr int B_BYTES = BN * 128;
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
  static constexpr int GSTART_OFF = PREFIX_OFF + 4 * (kMaxGroups + 1);
  static constexpr int SMEM_TOTAL = GSTART_OFF + 4 * (kMaxGroups + 1) + 1024;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "token tile");
  static_assert(COLS <= 512, "TMEM columns");
  static_assert(SMEM_TOTAL <= 232448, "shared memory");
};

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
};

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

// Warp-uniform bounded wait: every lane polls, the timeout decision is lane 0's.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* err) {
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

template <int MODE, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBfull, const Params p) {
  using C = Cfg<MODE, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + C::NBUF + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * C::NBUF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  int* prefix = reinterpret_cast<int*>(smem + C::PREFIX_OFF);
  int* gstart = reinterpret_cast<int*>(smem + C::GSTART_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (p.Mg + 127) / 128;
  const int KB = p.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA0);
    if (C::NA == 2) tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmBfull);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    // Batch boundaries, made safe: each clamped to [0, max_rows] and forced
    // non-decreasing (running max), so every batch lies inside the row
    // buffers whatever the caller passed; any change is flagged.
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
    // units per group: m_tiles x ceil(rows / BN); prefix over groups
    int carry = 0;
    if (lane == 0) prefix[0] = 0;
    for (int base = 0; base < p.n_groups; base += 32) {
      const int g = base + lane;
      int units = 0;
      if (g < p.n_groups) {
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = prefix[p.n_groups];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      // Weights are inputs no kernel of this sequence writes, and the unit
      // schedule comes from a grid two launches back: the first unit's weight
      // tiles are requested before waiting for the predecessor grid, whose
      // output (the token rows) is loaded only after the wait.
      int n_pre = 0;
      if ((int)blockIdx.x < total) {
        const Unit t = decode_unit<MODE, BN>(blockIdx.x, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const uint32_t bytes = C::NA * C::A_BYTES + ((t.nt + 31) / 32) * 4096;
        const int arow = t.g * p.Mg + t.mt * 128;
        n_pre = min(STAGES, t.kb1 - t.kb0);
        for (int i = 0; i < n_pre; ++i) {  // fresh ring: stages 0..n_pre-1 are free
          mbar_arrive_expect_tx(full_bar(i), bytes);
          armed |= 1u << i;
          const uint32_t sA = sbase + i * C::STAGE_BYTES;
          tma_load_2d(sA, &tmA0, full_bar(i), (t.kb0 + i) * 64, arow);
          if (C::NA == 2) tma_load_2d(sA + C::A_BYTES, &tmA1, full_bar(i), (t.kb0 + i) * 64, arow);
        }
      }
      pdl_wait();
      bool first = true;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        if (u + (int)gridDim.x >= total) pdl_trigger();  // this CTA's last unit
        const Unit t = decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int nchunks = (t.nt + 31) / 32;
        const uint32_t bytes = C::NA * C::A_BYTES + nchunks * 4096;
        const int arow = t.g * p.Mg + t.mt * 128;
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          const bool pre = first && kb - t.kb0 < n_pre;  // armed, weights already requested
          if (!pre) {
            if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(stage), bytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          const uint32_t sA = sbase + stage * C::STAGE_BYTES;
          if (!pre) {
            tma_load_2d(sA, &tmA0, full_bar(stage), kb * 64, arow);
            if (C::NA == 2) tma_load_2d(sA + C::A_BYTES, &tmA1, full_bar(stage), kb * 64, arow);
          }
          const uint32_t sB = sA + C::NA * C::A_BYTES;
          if (t.nt == BN)  // a full token tile: one box of BN rows
            tma_load_2d(sB, &tmBfull, full_bar(stage), kb * 64, t.r0);
          else
            for (int c = 0; c < nchunks; ++c)
              tma_load_2d(sB + c * 4096, &tmB, full_bar(stage), kb * 64, t.r0 + c * 32);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        first = false;
        if (!ok) break;
      }
      if ((int)blockIdx.x >= total) pdl_trigger();
      // wind down: every copy this thread started has landed before exit
      for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool issued = false;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x, ++it) {
        const Unit t = decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int n_mma = max(16, (t.nt + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(128, n_mma);
        const int buf = C::NBUF == 2 ? (it & 1) : 0;
        const uint32_t use = C::NBUF == 2 ? (uint32_t)(it >> 1) : (uint32_t)it;
        if (!mbar_wait(acce_bar(buf), (use & 1u) ^ 1u, abort_flag, p.err)) break;
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
            umma_bf16(d0, smem_desc_sw128(sA + kk * 32), bdesc, idesc, acc);
            if (C::NA == 2)
              umma_bf16(d0 + BN, smem_desc_sw128(sA + C::A_BYTES + kk * 32), bdesc, idesc, acc);
          }
          issued = true;
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(accf_bar(buf));
      }
      // wind down: every MMA this thread issued has completed before TMEM is freed
      if (issued) {
        umma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;  // the two warps of a quarter take alternate 16-column chunks
    int it = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
      const Unit t = decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
      const int buf = C::NBUF == 2 ? (it & 1) : 0;
      const uint32_t use = C::NBUF == 2 ? (uint32_t)(it >> 1) : (uint32_t)it;
      if (!mbar_wait_warp(accf_bar(buf), use & 1u, abort_flag, p.err)) break;
      tc_fence_after();
      const int m = t.mt * 128 + q * 32 + lane;  // weight row within the group
      const bool mvalid = m < p.Mg;
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * C::NACC * BN);
      for (int c0 = 16 * half; c0 < t.nt; c0 += 32) {
        uint32_t a[16], b[16];
        tmem_ld16(tb + c0, a);
        if (C::NA == 2) tmem_ld16(tb + BN + c0, b);
        tmem_ld_wait();
        if (mvalid) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col >= t.nt) break;
            const size_t row = (size_t)(t.r0 + col);
            const float v = __uint_as_float(a[j]);
            if (MODE == MODE_ROUTER) {
              const size_t chunk = (size_t)(t.kb0 / p.kb_per);
              static_cast<float*>(p.out)[(chunk * p.rows_single + row) * p.ldo + m] = v;
            } else if (MODE == MODE_GATEUP) {
              const float hval = silu_f32(v) * __uint_as_float(b[j]);
              static_cast<__nv_bfloat16*>(p.out)[row * p.ldo + m] = __float2bfloat16_rn(hval);
            } else {
              const float sc = p.row_scale ? p.row_scale[row] : 1.f;
              static_cast<__nv_bfloat16*>(p.out)[row * p.ldo + m] = __float2bfloat16_rn(v * sc);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// bf16 matrix [rows, inner] (row-major), boxes of box_rows x 64, 128-byte swizzle
bool make_tmap(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
               uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int BN, int STAGES>
cudaError_t launch_tc(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                      const CUtensorMap& bfull, const Params& p, long long max_units,
                      const char* name, cudaStream_t s) {
  using C = Cfg<MODE, BN, STAGES>;
  auto kern = tc_grouped_gemm<MODE, BN, STAGES>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const long long grid = max_units < num_sms() ? max_units : num_sms();
  if (grid <= 0) return cudaSuccess;
  ProfScope pr(name, s);
  (void)launch_kernel(kern, (unsigned)grid, kThreads, C::SMEM_TOTAL, s, a0, a1, b, bfull, p);
  return cudaGetLastError();
}

}  // namespace

// Rows of the workspace's permuted-row buffers: P rounded up so that every
// 32-row box a unit may touch lies inside the buffer.
int tc_row_capacity(int P) { return ((P + 31) / 32) * 32 + 256; }

cudaError_t launch_ffn_tc(const void* x_perm, const int32_t* offsets, int n_groups, int P,
                          int d, int I, double mean_rows, const void* Wg, const void* Wu,
                          const void* Wd, const float* slot_w, void* h, void* y_perm, int* err,
                          cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  const uint64_t cap = (uint64_t)tc_row_capacity(P);
  // Token tiles by mean batch size: 32 rows for decode-sized batches (deep
  // pipelines).  Above that, gate/up uses 128 rows while batches are a few
  // hundred rows (its two accumulators then fit twice in TMEM, so the epilogue
  // overlaps the next unit's MMAs) and 256 rows for larger batches (tensor
  // bound: the largest MMA); down uses 256 rows (fewest weight passes).
  const bool small = mean_rows <= 48.0;
  const int bn = small ? 32 : mean_rows <= 256.0 ? 128 : 256;
  // token operands: 32-row boxes for partial tiles, tile-high boxes for full ones
  CUtensorMap tg, tu, tx, txf, td, th, thf, thf2;
  if (!make_tmap(&tg, Wg, d, (uint64_t)n_groups * I, 128) ||
      !make_tmap(&tu, Wu, d, (uint64_t)n_groups * I, 128) ||
      !make_tmap(&tx, x_perm, d, cap, 32) || !make_tmap(&txf, x_perm, d, cap, bn) ||
      !make_tmap(&td, Wd, I, (uint64_t)n_groups * d, 128) || !make_tmap(&th, h, I, cap, 32) ||
      !make_tmap(&thf, h, I, cap, 32) || !make_tmap(&thf2, h, I, cap, 256))
    return cudaErrorInvalidValue;
  Params p1{offsets, n_groups, 0, I, d, h, I, nullptr, err, P};
  const long long u1 = (long long)((I + 127) / 128) * ((P + bn - 1) / bn + n_groups);
  cudaError_t e;
  if (small)
    e = launch_tc<MODE_GATEUP, 32, 6>(tg, tu, tx, txf, p1, u1, "ffn_gateup_tc", s);
  else if (bn == 128)
    e = launch_tc<MODE_GATEUP, 128, 4>(tg, tu, tx, txf, p1, u1, "ffn_gateup_tc", s);
  else
    e = launch_tc<MODE_GATEUP, 256, 3>(tg, tu, tx, txf, p1, u1, "ffn_gateup_tc", s);
  if (e != cudaSuccess) return e;
  const int bn2 = small ? 32 : 256;
  Params p2{offsets, n_groups, 0, d, I, y_perm, d, slot_w, err, P};
  const long long u2 = (long long)((d + 127) / 128) * ((P + bn2 - 1) / bn2 + n_groups);
  if (small) return launch_tc<MODE_DOWN, 32, 10>(td, td, th, thf, p2, u2, "ffn_down_tc", s);
  return launch_tc<MODE_DOWN, 256, 4>(td, td, th, thf2, p2, u2, "ffn_down_tc", s);
}

cudaError_t launch_router_logits_tc(const void* x, const void* Wr, int T, int d, int E,
                                    int ksplit, int kb_per, float* partial, int* err,
                                    cudaStream_t s) {
  if (T < 32 || E < 128 || ksplit < 1 || kb_per < 1) return cudaErrorInvalidValue;
  // a full 128-token box only exists when T >= 128; below that every unit is partial
  CUtensorMap ta, tb, tb128;
  if (!make_tmap(&ta, Wr, d, E, 128) || !make_tmap(&tb, x, d, T, 32) ||
      !make_tmap(&tb128, x, d, T, T >= 128 ? 128 : 32))
    return cudaErrorInvalidValue;
  Params p{nullptr, 1, T, E, d, partial, E, nullptr, err, T, ksplit, kb_per};
  const long long units = (long long)((E + 127) / 128) * ((T + 127) / 128) * ksplit;
  return launch_tc<MODE_ROUTER, 128, 6>(ta, ta, tb, tb128, p, units, "router_logits_tc", s);
}

}  // namespace moe
