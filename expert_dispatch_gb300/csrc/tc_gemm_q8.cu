// tc_gemm_q8.cu -- the expert FFN's grouped GEMMs with Q8_0 expert weights
// ("Distributed MoE" (tenzro docs), quantization table and compute-seam
// paragraph: experts block-quantized to Q8_0 -- 32-element blocks with one
// f16 scale -- and decoded by the holder's dequant path before Y = X * W^T).
//
// Same work units, MMA issue and epilogue as the bf16 kernel (tc_gemm.cu);
// what changes is how a weight tile reaches shared memory:
//   * the TMA producer loads, per 64-wide K block, the tile's int8 codes
//     (128 rows x 64 B), its f16 scales (2 blocks x 128 rows) and the token
//     rows into a "raw" stage (RS deep);
//   * converter warps decode codes into fp16 weights, scale * q rounded to
//     fp16, written straight into the 128-byte-swizzled K-major layout the
//     MMA descriptors expect, in a "converted" stage (CS deep), then make the
//     writes visible to the tensor core (fence.proxy.async) and signal;
//   * the MMA issuer (kind::f16 with fp16 operands, fp32 accumulation)
//     consumes converted weights and raw token rows and releases both stages
//     with tcgen05.commit.
// The operands are fp16 because the decode then costs one byte permute, one
// subtraction and one multiplication per two weights (packed half2), which
// keeps the converters ahead of HBM; token rows arrive in fp16 (converted
// from bf16 by the gather, exactly for values inside fp16's range) and the
// gate/up output H is written in fp16.  HBM moves 8.5 bits per weight.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {
namespace {

using tc::MODE_DOWN;
using tc::MODE_GATEUP;
using tc::Params;
using tc::Unit;
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kFirstConvWarp = 2 + tc::kEpiWarps;
constexpr int kThreadsQ8 = 32 * (2 + tc::kEpiWarps + kConvWarps);  // producer, MMA, epi, conv

template <int MODE, int BN, int RS, int CS>
struct CfgQ8 {
  static constexpr int NA = MODE == MODE_GATEUP ? 2 : 1;  // weight operands per K block
  static constexpr int QA_BYTES = 128 * 64;               // int8 codes of one weight tile
  static constexpr int SA_BYTES = 2 * 128 * 2;            // its f16 scales [2 blocks][128 rows]
  static constexpr int B_BYTES = BN * 128;                // token rows, fp16, 128-byte swizzle
  static constexpr int QA_OFF = B_BYTES;                  // offsets inside a raw stage
  static constexpr int SA_OFF = B_BYTES + NA * QA_BYTES;
  static constexpr int RAW_BYTES = (SA_OFF + NA * SA_BYTES + 1023) / 1024 * 1024;
  static constexpr int CA_BYTES = 128 * 64 * 2;           // one converted fp16 weight tile
  static constexpr int CONV_BYTES = NA * CA_BYTES;
  static constexpr int NACC = NA;
  static constexpr int NBUF = 2 * NACC * BN <= 512 ? 2 : 1;
  static constexpr int COLS = NBUF * NACC * BN;
  static constexpr int TMEM_COLS =
      COLS <= 32 ? 32 : COLS <= 64 ? 64 : COLS <= 128 ? 128 : COLS <= 256 ? 256 : 512;
  static constexpr int CONV_OFF = RS * RAW_BYTES;
  static constexpr int BAR_OFF = CONV_OFF + CS * CONV_BYTES;
  static constexpr int NBARS = 2 * RS + 2 * CS + 2 * NBUF + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int PREFIX_OFF = MISC_OFF + 16;
  static constexpr int GSTART_OFF = PREFIX_OFF + 4 * (tc::kMaxGroups + 1);
  static constexpr int SMEM_TOTAL = GSTART_OFF + 4 * (tc::kMaxGroups + 1) + 1024;
  static constexpr int CHUNKS_PER_THREAD = NA * 1024 / kConvThreads;  // 16-byte output chunks
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "token tile");
  static_assert(COLS <= 512, "TMEM columns");
  static_assert(RS <= 32, "raw stages tracked in a 32-bit mask");
  static_assert(NA * 1024 % kConvThreads == 0, "converter split");
  static_assert(SMEM_TOTAL <= 232448, "shared memory");
};

__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 8 int8 codes (one 8-byte word) times a scale, rounded to fp16, packed.
// Flipping the top bit of a code byte gives q + 128 in [0, 255]; a byte
// permute pairs two such bytes with the fp16 exponent of 1024, so each half
// reads 1024 + q + 128 exactly; subtracting 1152 leaves q exactly; the
// multiplication by the scale rounds once, to fp16.
__device__ __forceinline__ uint4 dequant8_f16(uint2 codes, __half2 scale2) {
  const uint32_t w0 = codes.x ^ 0x80808080u, w1 = codes.y ^ 0x80808080u;
  const __half2 magic = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
  uint32_t in[4] = {__byte_perm(w0, 0x64646464u, 0x4140u), __byte_perm(w0, 0x64646464u, 0x4342u),
                    __byte_perm(w1, 0x64646464u, 0x4140u), __byte_perm(w1, 0x64646464u, 0x4342u)};
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __half2 q2 = __hsub2(*reinterpret_cast<const __half2*>(&in[j]), magic);
    const __half2 v = __hmul2(q2, scale2);
    out[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

template <int MODE, int BN, int RS, int CS>
__global__ void __launch_bounds__(kThreadsQ8, 1)
    tc_grouped_gemm_q8(const __grid_constant__ CUtensorMap tmQ0,
                       const __grid_constant__ CUtensorMap tmQ1,
                       const __grid_constant__ CUtensorMap tmS0,
                       const __grid_constant__ CUtensorMap tmS1,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmBfull, const Params p) {
  using C = CfgQ8<MODE, BN, RS, CS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  auto raw_full = [&](int s) { return bar0 + 8u * s; };
  auto raw_empty = [&](int s) { return bar0 + 8u * (RS + s); };
  auto conv_full = [&](int s) { return bar0 + 8u * (2 * RS + s); };
  auto conv_empty = [&](int s) { return bar0 + 8u * (2 * RS + CS + s); };
  const uint32_t accf0 = bar0 + 8u * (2 * RS + 2 * CS);
  const uint32_t acce0 = accf0 + 8u * C::NBUF;
  const uint32_t drain_bar = acce0 + 8u * C::NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  int* prefix = reinterpret_cast<int*>(smem + C::PREFIX_OFF);
  int* gstart = reinterpret_cast<int*>(smem + C::GSTART_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (p.Mg + 127) / 128;
  const int KB = p.K / 64;
  const int sblocks = p.K / 32;  // scale blocks per weight row

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(raw_empty(s), 1);
    }
    for (int s = 0; s < CS; ++s) {
      mbar_init(conv_full(s), kConvWarps);
      mbar_init(conv_empty(s), 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(accf0 + 8u * b, 1);
      mbar_init(acce0 + 8u * b, tc::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ0);
    tma_prefetch_desc(&tmS0);
    if (C::NA == 2) {
      tma_prefetch_desc(&tmQ1);
      tma_prefetch_desc(&tmS1);
    }
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

  // weight codes and scales of one K block into a raw stage
  auto load_weights = [&](uint32_t raw, uint32_t bar, const Unit& t, int kb) {
    const int arow = t.g * p.Mg + t.mt * 128;
    const int srow = t.g * sblocks + kb * 2;
    tma_load_2d(raw + C::QA_OFF, &tmQ0, bar, kb * 64, arow);
    tma_load_2d(raw + C::SA_OFF, &tmS0, bar, t.mt * 128, srow);
    if (C::NA == 2) {
      tma_load_2d(raw + C::QA_OFF + C::QA_BYTES, &tmQ1, bar, kb * 64, arow);
      tma_load_2d(raw + C::SA_OFF + C::SA_BYTES, &tmS1, bar, t.mt * 128, srow);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      // the first unit's weight codes and scales are requested before waiting
      // for the predecessor grid (see tc_gemm.cu); token rows after the wait
      int n_pre = 0;
      if ((int)blockIdx.x < total) {
        const Unit t =
            tc::decode_unit<MODE, BN>(blockIdx.x, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const uint32_t bytes = C::NA * (C::QA_BYTES + C::SA_BYTES) + ((t.nt + 31) / 32) * 4096;
        n_pre = min(RS, t.kb1 - t.kb0);
        for (int i = 0; i < n_pre; ++i) {
          mbar_arrive_expect_tx(raw_full(i), bytes);
          armed |= 1u << i;
          load_weights(sbase + i * C::RAW_BYTES, raw_full(i), t, t.kb0 + i);
        }
      }
      pdl_wait();
      bool first = true;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        if (u + (int)gridDim.x >= total) pdl_trigger();  // this CTA's last unit
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int nchunks = (t.nt + 31) / 32;
        const uint32_t bytes = C::NA * (C::QA_BYTES + C::SA_BYTES) + nchunks * 4096;
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          const bool pre = first && kb - t.kb0 < n_pre;
          const uint32_t raw = sbase + stage * C::RAW_BYTES;
          if (!pre) {
            if (!mbar_wait(raw_empty(stage), phase ^ 1u, abort_flag, p.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(raw_full(stage), bytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            load_weights(raw, raw_full(stage), t, kb);
          }
          if (t.nt == BN)
            tma_load_2d(raw, &tmBfull, raw_full(stage), kb * 64, t.r0);
          else
            for (int c = 0; c < nchunks; ++c)
              tma_load_2d(raw + c * 4096, &tmB, raw_full(stage), kb * 64, t.r0 + c * 32);
          if (++stage == RS) {
            stage = 0;
            phase ^= 1u;
          }
        }
        first = false;
        if (!ok) break;
      }
      if ((int)blockIdx.x >= total) pdl_trigger();
      for (int s = 0; s < RS; ++s)
        if (armed & (1u << s)) tc::mbar_wait_drain(raw_full(s), (armed_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0;
      uint32_t kcount = 0;  // K blocks consumed so far (indexes both rings)
      bool issued = false;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x, ++it) {
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int n_mma = max(16, (t.nt + 15) & ~15);
        const uint32_t idesc = idesc_f16_f32(128, n_mma);
        const int buf = C::NBUF == 2 ? (it & 1) : 0;
        const uint32_t use = C::NBUF == 2 ? (uint32_t)(it >> 1) : (uint32_t)it;
        if (!mbar_wait(acce0 + 8u * buf, (use & 1u) ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(buf * C::NACC * BN);
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb, ++kcount) {
          const int rs = kcount % RS, cs = kcount % CS;
          if (!mbar_wait(conv_full(cs), (kcount / CS) & 1u, abort_flag, p.err) ||
              !mbar_wait(raw_full(rs), (kcount / RS) & 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sbase + C::CONV_OFF + cs * C::CONV_BYTES;
          const uint32_t sB = sbase + rs * C::RAW_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(sB + kk * 32);
            const uint32_t acc = (kb != t.kb0 || kk != 0) ? 1u : 0u;
            umma_bf16(d0, smem_desc_sw128(sA + kk * 32), bdesc, idesc, acc);
            if (C::NA == 2)
              umma_bf16(d0 + BN, smem_desc_sw128(sA + C::CA_BYTES + kk * 32), bdesc, idesc, acc);
          }
          issued = true;
          umma_commit(raw_empty(rs));
          umma_commit(conv_empty(cs));
        }
        if (!ok) break;
        umma_commit(accf0 + 8u * buf);
      }
      if (issued) {
        umma_commit(drain_bar);
        tc::mbar_wait_drain(drain_bar, 0, p.err);
      }
    }
  } else if (warp < kFirstConvWarp) {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    tc::epilogue_loop<MODE, BN, C::NACC, C::NBUF, true>(p, total, m_tiles, KB, prefix, gstart,
                                                        tmem_base, accf0, acce0, abort_flag, 2);
  } else {
    // ------------------------------------------------------------ converters
    // Thread ct owns 16-byte output column c = ct % 8 of rows (ct / 8) + 32 i
    // (i < 4 per weight operand): codes r*64 + c*8 .. +8 and scale block c/4
    // of row r become 8 fp16 values at row r, chunk c ^ (r % 8).  r % 8 and
    // c are fixed per thread, so every offset is a constant plus i * stride.
    const int ct = threadIdx.x - 32 * kFirstConvWarp;
    const int c = ct & 7, r0 = ct >> 3;
    const int code_off = C::QA_OFF + r0 * 64 + c * 8;
    const int scale_off = C::SA_OFF + ((c >> 2) * 128 + r0) * 2;
    const int dst_off = r0 * 128 + ((c ^ (r0 & 7)) << 4);
    uint32_t kcount = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
      for (int kb = t.kb0; kb < t.kb1; ++kb, ++kcount) {
        const int rs = kcount % RS, cs = kcount % CS;
        if (!tc::mbar_wait_warp(raw_full(rs), (kcount / RS) & 1u, abort_flag, p.err) ||
            !tc::mbar_wait_warp(conv_empty(cs), ((kcount / CS) & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint8_t* __restrict__ raw = smem + rs * C::RAW_BYTES;
        uint8_t* __restrict__ conv = smem + C::CONV_OFF + cs * C::CONV_BYTES;
        // all loads first (independent, so their latencies overlap), then decode and store
        uint2 codes[C::CHUNKS_PER_THREAD];
        __half sh[C::CHUNKS_PER_THREAD];
#pragma unroll
        for (int i = 0; i < C::CHUNKS_PER_THREAD; ++i) {
          const int op = i >> 2, rr = 32 * (i & 3);  // operand, row offset
          codes[i] = *reinterpret_cast<const uint2*>(raw + code_off + op * C::QA_BYTES + rr * 64);
          sh[i] = *reinterpret_cast<const __half*>(raw + scale_off + op * C::SA_BYTES + rr * 2);
        }
#pragma unroll
        for (int i = 0; i < C::CHUNKS_PER_THREAD; ++i) {
          const int op = i >> 2, rr = 32 * (i & 3);
          *reinterpret_cast<uint4*>(conv + dst_off + op * C::CA_BYTES + rr * 128) =
              dequant8_f16(codes[i], __halves2half2(sh[i], sh[i]));
        }
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(conv_full(cs));
      }
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

bool make_f16_map(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
                  uint32_t box_rows) {
  return make_tmap_2d(tm, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, inner, rows, 64, box_rows,
                      true);
}

// codes [n_groups * R, K] int8 in 128 x 64 boxes; scales [n_groups * K/32, R] f16 in 2 x 128 boxes
bool make_q8_maps(CUtensorMap* tq, CUtensorMap* ts, const Q8Weight& w, int n_groups, int R,
                  int K) {
  return make_tmap_2d(tq, w.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, (uint64_t)n_groups * R, 64,
                      128, false) &&
         make_tmap_2d(ts, w.scale, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, R,
                      (uint64_t)n_groups * (K / 32), 128, 2, false);
}

template <int MODE, int BN, int RS, int CS>
cudaError_t launch_q8(const CUtensorMap& q0, const CUtensorMap& q1, const CUtensorMap& s0,
                      const CUtensorMap& s1, const CUtensorMap& b, const CUtensorMap& bfull,
                      const Params& p, long long max_units, const char* name, cudaStream_t s) {
  using C = CfgQ8<MODE, BN, RS, CS>;
  auto kern = tc_grouped_gemm_q8<MODE, BN, RS, CS>;
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
  (void)launch_kernel(kern, (unsigned)grid, kThreadsQ8, C::SMEM_TOTAL, s, q0, q1, s0, s1, b,
                      bfull, p);
  return cudaGetLastError();
}

}  // namespace

// x_perm and h hold fp16 rows here (see the file comment).
cudaError_t launch_ffn_tc_q8(const void* x_perm, const int32_t* offsets, int n_groups, int P,
                             int d, int I, double mean_rows, const Q8Weight& Wg,
                             const Q8Weight& Wu, const Q8Weight& Wd, const float* slot_w,
                             void* h, void* y_perm, int* err, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  const uint64_t cap = (uint64_t)tc_row_capacity(P);
  const bool small = mean_rows <= 48.0;
  const int bn = small ? 32 : mean_rows <= 256.0 ? 128 : 256;
  CUtensorMap qg, sg, qu, su, qd, sd, tx, txf, th, thf2;
  if (!make_q8_maps(&qg, &sg, Wg, n_groups, I, d) || !make_q8_maps(&qu, &su, Wu, n_groups, I, d) ||
      !make_q8_maps(&qd, &sd, Wd, n_groups, d, I) || !make_f16_map(&tx, x_perm, d, cap, 32) ||
      !make_f16_map(&txf, x_perm, d, cap, bn) || !make_f16_map(&th, h, I, cap, 32) ||
      !make_f16_map(&thf2, h, I, cap, 256))
    return cudaErrorInvalidValue;
  Params p1{offsets, n_groups, 0, I, d, h, I, nullptr, err, P};
  const long long u1 = (long long)((I + 127) / 128) * ((P + bn - 1) / bn + n_groups);
  cudaError_t e;
  if (small)
    e = launch_q8<MODE_GATEUP, 32, 6, 2>(qg, qu, sg, su, tx, txf, p1, u1, "ffn_gateup_tc_q8", s);
  else if (bn == 128)
    e = launch_q8<MODE_GATEUP, 128, 4, 2>(qg, qu, sg, su, tx, txf, p1, u1, "ffn_gateup_tc_q8", s);
  else
    e = launch_q8<MODE_GATEUP, 256, 3, 2>(qg, qu, sg, su, tx, txf, p1, u1, "ffn_gateup_tc_q8", s);
  if (e != cudaSuccess) return e;
  const int bn2 = small ? 32 : 256;
  Params p2{offsets, n_groups, 0, d, I, y_perm, d, slot_w, err, P};
  const long long u2 = (long long)((d + 127) / 128) * ((P + bn2 - 1) / bn2 + n_groups);
  if (small)
    return launch_q8<MODE_DOWN, 32, 10, 3>(qd, qd, sd, sd, th, th, p2, u2, "ffn_down_tc_q8", s);
  return launch_q8<MODE_DOWN, 256, 4, 2>(qd, qd, sd, sd, th, thf2, p2, u2, "ffn_down_tc_q8", s);
}

}  // namespace moe
