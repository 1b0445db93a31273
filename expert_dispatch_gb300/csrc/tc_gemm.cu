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
//   * Work unit = (expert, MT-row weight block, token tile), MT = 128, or 256
//     for the decode-sized down GEMM (two 128-row boxes per stage and two
//     accumulators, as gate/up's two matrices); the order of units is
//     described at tc::decode_unit.
//   * Warp 0 lane 0 issues TMA loads (128-byte swizzle) into a STAGES-deep
//     shared-memory ring; warp 1 lane 0 issues tcgen05.mma (bf16 x bf16 ->
//     fp32 in TMEM) and commits each stage back to the loader; warps 2-9 read
//     the accumulators with tcgen05.ld and apply the epilogue (SwiGLU, row
//     scale) while, with two TMEM buffers, the next unit's MMAs run.
//   * Token rows are loaded in 32-row boxes for partial tiles and one
//     BN-row box for full tiles.
//   * Launched with programmatic dependent launch: the first unit's weight
//     tiles are requested before waiting for the previous kernel.
//   * Every wait is bounded (1 s); on expiry the CTA records a timeout in the
//     error word, drains its own copies and MMAs, frees TMEM and exits.
// Variants here: 32-token tiles (decode-sized batches, both FFN GEMMs),
// 256-token gate/up tiles (the largest batches) and the router.  The other
// large-batch FFN GEMMs run on SM pairs (tc_gemm_pair.cu); launch_ffn_tc
// picks per GEMM.
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
using tc::MODE_ROUTER;
using tc::Params;
using tc::Unit;
constexpr int kThreads = 32 * (2 + tc::kEpiWarps);  // producer, MMA, epilogue

template <int MODE, int BN, int STAGES, int MT = 128>
struct Cfg {
  // weight operands per stage: gate and up, or two 128-row blocks of one
  // matrix when a unit spans MT = 256 weight rows
  static constexpr int NA = MODE == MODE_GATEUP || MT == 256 ? 2 : 1;
  // the second operand's first row, relative to the unit's
  static constexpr int A1_ROW = MODE == MODE_GATEUP ? 0 : 128;
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
  static constexpr int GSTART_OFF = PREFIX_OFF + 4 * (tc::kMaxGroups + 1);
  static constexpr int SMEM_TOTAL = GSTART_OFF + 4 * (tc::kMaxGroups + 1) + 1024;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "token tile");
  static_assert(MT == 128 || (MT == 256 && MODE != MODE_GATEUP), "weight rows per unit");
  static_assert(COLS <= 512, "TMEM columns");
  static_assert(SMEM_TOTAL <= 232448, "shared memory");
};

template <int MODE, int BN, int STAGES, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBfull, const Params p) {
  using C = Cfg<MODE, BN, STAGES, MT>;
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
  const int m_tiles = (p.Mg + MT - 1) / MT;
  const int KB = p.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(accf0 + 8u * b, 1);
      mbar_init(acce0 + 8u * b, tc::kEpiWarps);
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
  if (warp == 2) tc::build_schedule<MODE, BN>(p, m_tiles, prefix, gstart);
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
        const Unit t =
            tc::decode_unit<MODE, BN>(blockIdx.x, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const uint32_t bytes = C::NA * C::A_BYTES + ((t.nt + 31) / 32) * 4096;
        const int arow = tc::weight_mat(p, t.g) * p.Mg + t.mt * MT;
        n_pre = min(STAGES, t.kb1 - t.kb0);
        for (int i = 0; i < n_pre; ++i) {  // fresh ring: stages 0..n_pre-1 are free
          mbar_arrive_expect_tx(full_bar(i), bytes);
          armed |= 1u << i;
          const uint32_t sA = sbase + i * C::STAGE_BYTES;
          tma_load_2d(sA, &tmA0, full_bar(i), (t.kb0 + i) * 64, arow);
          if (C::NA == 2)
            tma_load_2d(sA + C::A_BYTES, &tmA1, full_bar(i), (t.kb0 + i) * 64, arow + C::A1_ROW);
        }
      }
      pdl_wait();
      bool first = true;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        if (u + (int)gridDim.x >= total) pdl_trigger();  // this CTA's last unit
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int nchunks = (t.nt + 31) / 32;
        const uint32_t bytes = C::NA * C::A_BYTES + nchunks * 4096;
        const int arow = tc::weight_mat(p, t.g) * p.Mg + t.mt * MT;
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
            if (C::NA == 2)
              tma_load_2d(sA + C::A_BYTES, &tmA1, full_bar(stage), kb * 64, arow + C::A1_ROW);
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
        if (armed & (1u << s)) tc::mbar_wait_drain(full_bar(s), (armed_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool issued = false;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x, ++it) {
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int n_mma = max(16, (t.nt + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(128, n_mma);
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
        umma_commit(accf0 + 8u * buf);
      }
      // wind down: every MMA this thread issued has completed before TMEM is freed
      if (issued) {
        umma_commit(drain_bar);
        tc::mbar_wait_drain(drain_bar, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    tc::epilogue_loop<MODE, BN, C::NACC, C::NBUF, false, 1, MT>(
        p, total, m_tiles, KB, prefix, gstart, tmem_base, accf0, acce0, abort_flag, 2, blockIdx.x,
        gridDim.x, 0);
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
  return make_tmap_2d(tm, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, rows, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE, int BN, int STAGES, int MT = 128>
cudaError_t launch_tc(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                      const CUtensorMap& bfull, const Params& p, long long max_units,
                      const char* name, cudaStream_t s) {
  using C = Cfg<MODE, BN, STAGES, MT>;
  auto kern = tc_grouped_gemm<MODE, BN, STAGES, MT>;
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

bool make_tmap_2d(CUtensorMap* tm, const void* base, CUtensorMapDataType dtype, int elsize,
                  uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                  CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * (uint64_t)elsize};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, dtype, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of the workspace's permuted-row buffers: P rounded up so that every
// 32-row box a unit may touch lies inside the buffer.
int tc_row_capacity(int P) { return ((P + 31) / 32) * 32 + 256; }

cudaError_t launch_ffn_tc(const void* x_perm, const int32_t* offsets, int n_groups, int P,
                          int d, int I, double mean_rows, const void* Wg, const void* Wu,
                          const void* Wd, const float* slot_w, void* h, void* y_perm, int* err,
                          cudaStream_t s, int n_mats, const int32_t* group_slot) {
  if (P == 0) return cudaSuccess;
  const uint64_t cap = (uint64_t)tc_row_capacity(P);
  // Token tiles by mean batch size: 32 rows for decode-sized batches (one SM
  // per tile, deep pipelines).  Larger batches: gate/up with 160-row tiles
  // while batches are up to a few hundred rows (a batch of 95-160 rows is one
  // tile, so its weights pass once), 256 beyond (tensor bound: the largest
  // MMA); down always with 256-row tiles (fewer tiles per batch, so fewer
  // passes over its weights: measured faster than 160 on prefill batches of
  // ~140 rows).  Large tiles run on SM pairs (tc_gemm_pair.cu), except gate/up
  // with 256-row tiles: its two accumulators fill TMEM, and the pair's single
  // buffer, released only when both CTAs' epilogues are done with it, stalls
  // the MMA longer than on one SM, which measured faster there.
  const bool small = mean_rows <= 48.0;
  const int bn = small ? 32 : mean_rows <= 256.0 ? 160 : 256;
  if (n_mats <= 0) n_mats = n_groups;
  CUtensorMap tg, tu, td;
  if (!make_tmap(&tg, Wg, d, (uint64_t)n_mats * I, 128) ||
      !make_tmap(&tu, Wu, d, (uint64_t)n_mats * I, 128) ||
      !make_tmap(&td, Wd, I, (uint64_t)n_mats * d, 128))
    return cudaErrorInvalidValue;
  Params p1{offsets, n_groups, 0, I, d, h, I, nullptr, err, P, 0, 0, group_slot};
  Params p2{offsets, n_groups, 0, d, I, y_perm, d, slot_w, err, P, 0, 0, group_slot};
  const long long tiles = (long long)(P + bn - 1) / bn + n_groups;
  if (small) {
    // token operands: 32-row boxes (a tile is one box)
    CUtensorMap tx, th;
    if (!make_tmap(&tx, x_perm, d, cap, 32) || !make_tmap(&th, h, I, cap, 32))
      return cudaErrorInvalidValue;
    const cudaError_t e = launch_tc<MODE_GATEUP, 32, 6>(tg, tu, tx, tx, p1, (I + 127) / 128 * tiles,
                                                        "ffn_gateup_tc", s);
    if (e != cudaSuccess) return e;
    // down: units of 256 weight rows (two 128-row blocks per stage, as gate/up's
    // two matrices), so each stage carries 32 KB of weights
    return launch_tc<MODE_DOWN, 32, 6, 256>(td, td, th, th, p2, (d + 255) / 256 * tiles,
                                            "ffn_down_tc", s);
  }
  // SM pairs: one token box per CTA and K block, (i + 1) * 16 rows high
  PairTokenMaps pxm, phm;
  for (int i = 0; i < 8; ++i)
    if ((i < bn / 32 && !make_tmap(&pxm.box[i], x_perm, d, cap, 16 * (i + 1))) ||
        !make_tmap(&phm.box[i], h, I, cap, 16 * (i + 1)))
      return cudaErrorInvalidValue;
  cudaError_t e;
  if (bn == 160) {
    e = launch_gateup_pair(tg, tu, pxm, p1, P, n_groups, s);
  } else {  // one SM per tile: 32-row boxes for partial tiles, one 256-row box for full ones
    CUtensorMap tx, txf;
    if (!make_tmap(&tx, x_perm, d, cap, 32) || !make_tmap(&txf, x_perm, d, cap, 256))
      return cudaErrorInvalidValue;
    e = launch_tc<MODE_GATEUP, 256, 3>(tg, tu, tx, txf, p1, (I + 127) / 128 * tiles,
                                       "ffn_gateup_tc", s);
  }
  if (e != cudaSuccess) return e;
  return launch_down_pair(td, phm, p2, P, n_groups, s);
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

// Self-check of the bounded waits that every tcgen05 kernel here uses: one CTA
// waits on an mbarrier whose phase nothing completes.  The wait has to give up
// after kWaitLimitNs, record kErrTimeout in *err and return, and the kernel
// then ends normally, so the context stays usable.
//   which 0: the single-thread wait (mbar_wait)
//   which 1: the warp-uniform wait (mbar_wait_warp)
//   which 2: the wind-down wait that ignores the abort flag (mbar_wait_drain)
//   which 3: a warp-uniform wait and a single-thread wait sharing one abort
//            flag: whichever expires first has to release the other
__global__ void __launch_bounds__(64, 1) bounded_wait_check_kernel(int which, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const uint32_t b = smem_u32(&bar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (which == 0) {
    if (threadIdx.x == 0) mbar_wait(b, 0, &abort_flag, err);
  } else if (which == 1) {
    if (warp == 0) tc::mbar_wait_warp(b, 0, &abort_flag, err);
  } else if (which == 2) {
    if (threadIdx.x == 0) tc::mbar_wait_drain(b, 0, err);
  } else {
    if (warp == 0) tc::mbar_wait_warp(b, 0, &abort_flag, err);
    else if (lane == 0) mbar_wait(b, 0, &abort_flag, err);
  }
  __syncthreads();
}

cudaError_t launch_bounded_wait_check(int which, int* err, cudaStream_t s) {
  if (which < 0 || which > 3) return cudaErrorInvalidValue;
  ProfScope pr("bounded_wait_check", s);
  count_launch();
  bounded_wait_check_kernel<<<1, 64, 0, s>>>(which, err);
  return cudaGetLastError();
}

}  // namespace moe
