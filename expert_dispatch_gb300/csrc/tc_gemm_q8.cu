// tc_gemm_q8.cu -- the expert FFN's grouped GEMMs with Q8_0 expert weights
// ("Distributed MoE" (tenzro docs), quantization table and compute-seam
// paragraph: experts block-quantized to Q8_0 -- 32-element blocks with one
// f16 scale -- and decoded by the holder's dequant path before Y = X * W^T).
//
// Same work units, MMA shape and epilogue as the bf16 kernel (tc_gemm.cu);
// what changes is how a weight tile reaches the tensor core.  Per 64-wide K
// block of a unit:
//   * the weight loader (warp 0) brings the tile's int8 codes and f16 scales
//     into a weight stage (WS deep), two K blocks per stage: 128 rows x 128 B
//     of codes (128-byte swizzle) and 4 scale blocks x 128 rows, so each copy
//     moves whole 128-byte code rows (with one 64-byte row per K block the
//     down GEMM, one operand per stage, measured ~10 % slower);
//   * the token loader (warp 2) brings the unit's token rows (fp16, 128-byte
//     swizzle) into a token stage (TS deep);
//   * converter warps read the codes and scales into registers, decode the
//     stage's first K block and hand the weight stage back (each lane first
//     fences its reads against the loader's next TMA copy into the stage:
//     different proxies), then decode the second:
//     scale * q rounded to fp16.
//     The MMA takes its M-side operand from tensor memory (one weight row per
//     TMEM lane, two 16-bit K elements per 32-bit column), so each converter
//     thread owns one row of its warp's lane quarter and writes it with
//     tcgen05.st into a converted stage (CS deep, in TMEM);
//   * the MMA issuer (kind::f16, fp16 operands, fp32 accumulation) consumes a
//     converted stage and a token stage and releases both with
//     tcgen05.commit.  With 32-token tiles an MMA is so short that a single
//     issuing thread cannot keep up with the weight stream (one thread
//     issues at most one MMA per ~45 cycles, and each K block also costs it
//     two waits, a fence and two commits), so NI issuers (2 for gate/up, 4
//     for down) take K block j of each unit when j % NI is theirs, into NI
//     partial accumulators that the epilogue adds.  The large-tile gate/up
//     has no TMEM for partial sets; there two issuers split the operands
//     instead (gate MMAs on one thread, up MMAs on the other), because each
//     issuer's waits stall it until its own MMAs drain.
// A weight stage is thus held only from its TMA until the converters have
// decoded its first K block, so the in-flight depth of the weight stream does
// not shrink by the MMA latency; the weight loader never waits for the predecessor grid
// (weights are never written by the kernel just before; the token rows are,
// so the token loader waits).  The 128-byte swizzle puts 16-byte chunk j of
// code row r at chunk j ^ (r % 8), so a warp's 32 rows read one chunk each
// in the minimum four shared-memory wavefronts.
// The operands are fp16 because the decode then costs one byte permute, one
// subtraction and one multiplication per two weights (packed half2); token
// rows arrive in fp16 (converted from bf16 by the gather, exactly for values
// inside fp16's range) and the gate/up output H is written in fp16.  HBM
// moves 8.5 bits per weight.
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
constexpr int kFirstEpiWarp = 3;  // warps 0-2: weight loader, MMA issuer, token loader
constexpr int kFirstConvWarp = kFirstEpiWarp + tc::kEpiWarps;
constexpr int kIssuer2 = kFirstConvWarp + kConvWarps;  // issuers 2 .. NI: warps kIssuer2 ..
constexpr int threads_q8(int NI) { return 32 * (kIssuer2 + NI - 1); }

template <int MODE, int BN, int WS, int TS, int CS, int NI, bool OPS>
struct CfgQ8 {
  static constexpr int NA = MODE == MODE_GATEUP ? 2 : 1;  // weight operands per K block
  // NI issuers either split the K blocks of a unit (each into partial
  // accumulators of its own, added by the epilogue) or, with OPS, take one
  // operand each (gate / up) of every K block
  static constexpr int NPART = OPS ? 1 : NI;  // partial accumulator sets
  static constexpr int NCB = OPS ? 2 : 1;     // converted-stage barrier pairs per stage
  static constexpr int QA_BYTES = 128 * 128;  // int8 codes of a weight tile: 128 rows x two K blocks
  static constexpr int SA_BYTES = 4 * 128 * 2;  // its f16 scales [4 blocks][128 rows]
  static constexpr int SA_OFF = NA * QA_BYTES;            // scales inside a weight stage
  static constexpr int W_TX = NA * (QA_BYTES + SA_BYTES);  // bytes one weight stage receives
  static constexpr int W_BYTES = (W_TX + 1023) / 1024 * 1024;
  static constexpr int B_BYTES = BN * 128;                // token rows of one K block
  static constexpr int T_OFF = WS * W_BYTES;
  static constexpr int NACC = NA;
  // converter warps per K block: gate/up needs all of them (two operands x
  // four lane quarters); down's single operand takes four, so two groups of
  // four convert alternate K blocks concurrently
  static constexpr int CONV_PER_BLOCK = NA == 2 ? kConvWarps : kConvWarps / 2;
  static constexpr int A_COLS = NA * 32 * CS;             // TMEM columns of the converted ring
  // converter warps arriving on one converted-stage barrier
  static constexpr int CONV_ARRIVALS = OPS ? kConvWarps / 2 : CONV_PER_BLOCK;
  static constexpr int NBUF = 2 * NPART * NACC * BN + A_COLS <= 512 ? 2 : 1;
  static constexpr int ACC_COLS = NBUF * NPART * NACC * BN;  // [buffer][part][operand][BN]
  static constexpr int COLS = ACC_COLS + A_COLS;
  static constexpr int TMEM_COLS =
      COLS <= 32 ? 32 : COLS <= 64 ? 64 : COLS <= 128 ? 128 : COLS <= 256 ? 256 : 512;
  static constexpr int BAR_OFF = T_OFF + TS * B_BYTES;
  static constexpr int NBARS = 2 * WS + 2 * TS + 2 * CS * NCB + 2 * NBUF + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int PREFIX_OFF = MISC_OFF + 16;
  static constexpr int GSTART_OFF = PREFIX_OFF + 4 * (tc::kMaxGroups + 1);
  static constexpr int SMEM_TOTAL = GSTART_OFF + 4 * (tc::kMaxGroups + 1) + 1024;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "token tile");
  static_assert(COLS <= 512, "TMEM columns");
  static_assert(WS <= 32 && TS <= 32, "stages in flight tracked in 32-bit masks");
  static_assert(NI >= 1 && NI <= 4, "issuers");
  static_assert(!OPS || (NA == 2 && NI == 2), "operand split: one issuer per gate/up operand");
  // K split: K block j goes to issuer j % NI and to token / converted stage
  // j % TS / j % CS.  With TS and CS multiples of NI every stage is only ever
  // taken by one issuer, so no issuer can run a full phase ahead of a stage
  // another issuer still holds (its parity wait would then see the older
  // phase complete).  Operand split: both issuers take every token stage, which
  // is refilled only after both have released it, so neither can run a phase
  // ahead; each converted-stage barrier has one issuer.
  static_assert(OPS || (TS % NI == 0 && CS % NI == 0), "ring stages per issuer");
  static_assert(SMEM_TOTAL <= 232448, "shared memory");
};

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

template <int MODE, int BN, int WS, int TS, int CS, int NI, bool OPS>
__global__ void __launch_bounds__(threads_q8(NI), 1)
    tc_grouped_gemm_q8(const __grid_constant__ CUtensorMap tmQ0,
                       const __grid_constant__ CUtensorMap tmQ1,
                       const __grid_constant__ CUtensorMap tmS0,
                       const __grid_constant__ CUtensorMap tmS1,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmBfull, const Params p) {
  using C = CfgQ8<MODE, BN, WS, TS, CS, NI, OPS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  auto w_full = [&](int s) { return bar0 + 8u * s; };
  auto w_empty = [&](int s) { return bar0 + 8u * (WS + s); };
  auto t_full = [&](int s) { return bar0 + 8u * (2 * WS + s); };
  auto t_empty = [&](int s) { return bar0 + 8u * (2 * WS + TS + s); };
  // converted stage s of operand set b (b = the operand with OPS, else 0)
  auto conv_full = [&](int s, int b) { return bar0 + 8u * (2 * WS + 2 * TS + s * C::NCB + b); };
  auto conv_empty = [&](int s, int b) {
    return bar0 + 8u * (2 * WS + 2 * TS + (CS + s) * C::NCB + b);
  };
  const uint32_t accf0 = bar0 + 8u * (2 * WS + 2 * TS + 2 * CS * C::NCB);
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
    for (int s = 0; s < WS; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(w_empty(s), C::CONV_PER_BLOCK);
    }
    for (int s = 0; s < TS; ++s) {
      mbar_init(t_full(s), 1);
      mbar_init(t_empty(s), OPS ? 2 : 1);
    }
    for (int s = 0; s < CS; ++s)
      for (int b = 0; b < C::NCB; ++b) {
        mbar_init(conv_full(s, b), C::CONV_ARRIVALS);
        mbar_init(conv_empty(s, b), 1);
      }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(accf0 + 8u * b, NI);
      mbar_init(acce0 + 8u * b, tc::kEpiWarps);
    }
    mbar_init(drain_bar, NI);
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

  if (warp == 0) {
    // ------------------------------------------------------------ weight loader
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int mat = tc::weight_mat(p, t.g);
        const int arow = mat * p.Mg + t.mt * 128;
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; kb += 2) {  // a stage holds K blocks kb, kb + 1
          if (!mbar_wait(w_empty(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t bar = w_full(stage), w = sbase + stage * C::W_BYTES;
          mbar_arrive_expect_tx(bar, C::W_TX);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          const int srow = mat * sblocks + kb * 2;
          tma_load_2d(w, &tmQ0, bar, kb * 64, arow);
          tma_load_2d(w + C::SA_OFF, &tmS0, bar, t.mt * 128, srow);
          if (C::NA == 2) {
            tma_load_2d(w + C::QA_BYTES, &tmQ1, bar, kb * 64, arow);
            tma_load_2d(w + C::SA_OFF + C::SA_BYTES, &tmS1, bar, t.mt * 128, srow);
          }
          if (++stage == WS) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // wind down: every copy this thread started has landed before exit
      for (int s = 0; s < WS; ++s)
        if (armed & (1u << s)) tc::mbar_wait_drain(w_full(s), (armed_parity >> s) & 1u, p.err);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ token loader
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      pdl_wait();  // token rows come from the previous kernel
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x) {
        if (u + (int)gridDim.x >= total) pdl_trigger();  // this CTA's last unit
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int nchunks = (t.nt + 31) / 32;
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(t_empty(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t bar = t_full(stage), sB = sbase + C::T_OFF + stage * C::B_BYTES;
          mbar_arrive_expect_tx(bar, nchunks * 4096);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (t.nt == BN)  // a full token tile: one box of BN rows
            tma_load_2d(sB, &tmBfull, bar, kb * 64, t.r0);
          else
            for (int c = 0; c < nchunks; ++c)
              tma_load_2d(sB + c * 4096, &tmB, bar, kb * 64, t.r0 + c * 32);
          if (++stage == TS) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if ((int)blockIdx.x >= total) pdl_trigger();
      for (int s = 0; s < TS; ++s)
        if (armed & (1u << s)) tc::mbar_wait_drain(t_full(s), (armed_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1 || warp >= kIssuer2) {
    // ------------------------------------------------------------ MMA issuer(s)
    // K split: issuer i takes the K blocks kb of each unit with
    // (kb - kb0) % NI == i into its own partial accumulators.  Operand split:
    // issuer i issues operand i's MMAs of every K block.  Every issuer commits
    // each unit's accumulators (accf counts NI arrivals) and the final drain.
    // A thread that has issued tcgen05.mma and then waits on an mbarrier (or
    // reads shared memory at all) stalls until its queued MMAs have drained:
    // ~260 SM cycles per K block, measured with back-to-back M=128 K=16 MMAs,
    // against 4 x N/2 cycles of MMA work per operand.  Two issuers fill each
    // other's stalls: the operand split made the 192-token gate/up ~6 % faster.
    const int me = warp == 1 ? 0 : warp - kIssuer2 + 1;
    if (lane == 0 && me < NI) {
      int it = 0;
      uint32_t kcount = 0;  // K blocks seen so far (indexes the token and converted rings)
      for (int u = blockIdx.x; u < total && !*abort_flag; u += gridDim.x, ++it) {
        const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
        const int n_mma = max(16, (t.nt + 15) & ~15);
        const uint32_t idesc = idesc_f16_f32(128, n_mma);
        const int buf = C::NBUF == 2 ? (it & 1) : 0;
        const uint32_t use = C::NBUF == 2 ? (uint32_t)(it >> 1) : (uint32_t)it;
        if (!mbar_wait(acce0 + 8u * buf, (use & 1u) ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d0 =
            OPS ? tmem_base + (uint32_t)((buf * C::NACC + me) * BN)
                : tmem_base + (uint32_t)((buf * NI + me) * C::NACC * BN);
        const int cb = OPS ? me : 0;
        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb, ++kcount) {
          if (!OPS && (kb - t.kb0) % NI != me) continue;
          const int ts = kcount % TS, cs = kcount % CS;
          if (!mbar_wait(conv_full(cs, cb), (kcount / CS) & 1u, abort_flag, p.err) ||
              !mbar_wait(t_full(ts), (kcount / TS) & 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sB = sbase + C::T_OFF + ts * C::B_BYTES;
          // operand op of converted stage cs: columns ACC_COLS + (cs * NA + op) * 32,
          // 8 columns per K=16 step
          const uint32_t tA =
              tmem_base + (uint32_t)(C::ACC_COLS + cs * C::NA * 32 + (OPS ? me * 32 : 0));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(sB + kk * 32);
            const uint32_t acc = (kb - t.kb0 >= (OPS ? 1 : NI) || kk != 0) ? 1u : 0u;
            umma_f16_ts(d0, tA + kk * 8, bdesc, idesc, acc);
            if (C::NA == 2 && !OPS) umma_f16_ts(d0 + BN, tA + 32 + kk * 8, bdesc, idesc, acc);
          }
          umma_commit(t_empty(ts));
          umma_commit(conv_empty(cs, cb));
        }
        if (!ok) break;
        umma_commit(accf0 + 8u * buf);
      }
      if ((int)blockIdx.x < total) {  // every issuer arrives, whether or not it issued
        umma_commit(drain_bar);
        tc::mbar_wait_drain(drain_bar, 0, p.err);
      }
    }
  } else if (warp < kFirstConvWarp) {
    // ------------------------------------------------------------ epilogue (warps 3..10)
    tc::epilogue_loop<MODE, BN, C::NACC, C::NBUF, true, C::NPART>(p, total, m_tiles, KB, prefix,
                                                            gstart, tmem_base, accf0, acce0,
                                                            abort_flag, kFirstEpiWarp,
                                                            blockIdx.x, gridDim.x, 0);
  } else {
    // ------------------------------------------------------------ converters
    // Warp w may write only TMEM lanes 32 (w % 4) .. +31, so thread (w, lane)
    // owns weight row r = 32 (w % 4) + lane: per weight stage it reads its
    // row's 128 codes (two K blocks) and four scales, hands the stage back,
    // then decodes and writes one converted K block at a time.  Gate/up: the
    // first four converter warps decode operand 0, the other four operand 1.
    // Down: the first four take the even weight stages of this CTA's
    // sequence, the other four the odd ones, so two stages are in conversion
    // at once (a down stage is half the bytes of a gate/up one, and one at a
    // time left the converters short of the weight stream).
    constexpr int NCH = 8;  // 16-byte code chunks per thread: a 128-weight row
    const int cw = warp - kFirstConvWarp;
    const int q = warp & 3, r = q * 32 + lane;
    const int op = C::NA == 2 ? cw >> 2 : 0;
    const int cb = OPS ? op : 0;  // converted-stage barriers this warp uses
    const uint32_t group = C::NA == 2 ? 0u : (uint32_t)(cw >> 2);  // down: stage parity
    const int swz = r & 7;  // 128-byte swizzle: chunk j of code row r sits at j ^ (r % 8)
    const int code_off = op * C::QA_BYTES + r * 128;
    const int scale_off = C::SA_OFF + op * C::SA_BYTES + r * 2;  // + scale block * 256
    const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(C::ACC_COLS + op * 32);
    uint32_t kcount = 0, wcount = 0;  // K blocks and weight stages seen so far
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit t = tc::decode_unit<MODE, BN>(u, prefix, gstart, p.n_groups, m_tiles, KB, p);
      for (int kb = t.kb0; kb < t.kb1 && ok; kb += 2, ++wcount) {
        const int nk = min(2, t.kb1 - kb);  // K blocks in this stage
        if (C::NA == 1 && (wcount & 1u) != group) {
          kcount += nk;
          continue;
        }
        const int ws = wcount % WS;
        if (!tc::mbar_wait_warp(w_full(ws), (wcount / WS) & 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint8_t* w = smem + ws * C::W_BYTES;
        uint4 codes[NCH];
        __half sh[NCH / 2];
#pragma unroll
        for (int i = 0; i < NCH; ++i)
          codes[i] = *reinterpret_cast<const uint4*>(w + code_off + ((i ^ swz) << 4));
#pragma unroll
        for (int b = 0; b < NCH / 2; ++b)
          sh[b] = *reinterpret_cast<const __half*>(w + scale_off + b * 256);
        // The stage goes back to the loader once its first K block is decoded
        // (every code and scale is in registers by then).  The loader's next
        // copy into it is an async-proxy write, so every lane first orders its
        // reads before it with a proxy fence: without one, rows of a tile were
        // seen decoded from the next stage's data under light HBM load.  Placed
        // after the first block's decode, the fence waits for nothing.
        auto hand_back = [&] {
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(w_empty(ws));
        };
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h >= nk) break;
          const int cs = kcount % CS;
          if (!tc::mbar_wait_warp(conv_empty(cs, cb), ((kcount / CS) & 1u) ^ 1u, abort_flag,
                                  p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t o[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 4 * h + i;  // code chunk: 16 codes, scale block c / 2
            const __half2 s2 = __halves2half2(sh[c >> 1], sh[c >> 1]);
            const uint4 lo = dequant8_f16(make_uint2(codes[c].x, codes[c].y), s2);
            const uint4 hi = dequant8_f16(make_uint2(codes[c].z, codes[c].w), s2);
            o[8 * i + 0] = lo.x;
            o[8 * i + 1] = lo.y;
            o[8 * i + 2] = lo.z;
            o[8 * i + 3] = lo.w;
            o[8 * i + 4] = hi.x;
            o[8 * i + 5] = hi.y;
            o[8 * i + 6] = hi.z;
            o[8 * i + 7] = hi.w;
          }
          tmem_st32(t_row + (uint32_t)(cs * C::NA * 32), o);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(conv_full(cs, cb));
          ++kcount;
          if (h == 0) hand_back();
        }
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
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

// codes [n_groups * R, K] int8 in 128 x 128 boxes (two K blocks), 128-byte
// swizzle; scales [n_groups * K/32, R] f16 in 4 x 128 boxes
bool make_q8_maps(CUtensorMap* tq, CUtensorMap* ts, const Q8Weight& w, int n_groups, int R,
                  int K) {
  return make_tmap_2d(tq, w.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, (uint64_t)n_groups * R, 128,
                      128, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_tmap_2d(ts, w.scale, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, R,
                      (uint64_t)n_groups * (K / 32), 128, 4, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int MODE, int BN, int WS, int TS, int CS, int NI, bool OPS = false>
cudaError_t launch_q8(const CUtensorMap& q0, const CUtensorMap& q1, const CUtensorMap& s0,
                      const CUtensorMap& s1, const CUtensorMap& b, const CUtensorMap& bfull,
                      const Params& p, long long max_units, const char* name, cudaStream_t s) {
  using C = CfgQ8<MODE, BN, WS, TS, CS, NI, OPS>;
  auto kern = tc_grouped_gemm_q8<MODE, BN, WS, TS, CS, NI, OPS>;
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
  (void)launch_kernel(kern, (unsigned)grid, threads_q8(NI), C::SMEM_TOTAL, s, q0, q1, s0, s1, b,
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
  // gate/up keeps two accumulators per unit beside the converted ring in
  // TMEM: 192-token tiles leave room for a two-deep ring (2 x 192 + 2 x 64
  // columns), and keep prefill batches of up to 192 rows in one tile (with
  // 128-token tiles, batches of ~140 rows split into a second tile of a few
  // rows whose N=16 MMAs are issue-bound: measured ~15 % slower)
  const int bn = small ? 32 : 192;
  const int bn2 = small ? 32 : 256;
  CUtensorMap qg, sg, qu, su, qd, sd, tx, txf, th, thf2;
  if (!make_q8_maps(&qg, &sg, Wg, n_groups, I, d) || !make_q8_maps(&qu, &su, Wu, n_groups, I, d) ||
      !make_q8_maps(&qd, &sd, Wd, n_groups, d, I) || !make_f16_map(&tx, x_perm, d, cap, 32) ||
      !make_f16_map(&txf, x_perm, d, cap, bn) || !make_f16_map(&th, h, I, cap, 32) ||
      !make_f16_map(&thf2, h, I, cap, bn2))
    return cudaErrorInvalidValue;
  Params p1{offsets, n_groups, 0, I, d, h, I, nullptr, err, P};
  const long long u1 = (long long)((I + 127) / 128) * ((P + bn - 1) / bn + n_groups);
  const char* n1 = "ffn_gateup_tc_q8";
  const cudaError_t e =
      small ? launch_q8<MODE_GATEUP, 32, 5, 8, 4, 2>(qg, qu, sg, su, tx, txf, p1, u1, n1, s)
            : launch_q8<MODE_GATEUP, 192, 3, 4, 2, 2, true>(qg, qu, sg, su, tx, txf, p1, u1, n1, s);
  if (e != cudaSuccess) return e;
  Params p2{offsets, n_groups, 0, d, I, y_perm, d, slot_w, err, P};
  const long long u2 = (long long)((d + 127) / 128) * ((P + bn2 - 1) / bn2 + n_groups);
  const char* n2 = "ffn_down_tc_q8";
  return small ? launch_q8<MODE_DOWN, 32, 10, 8, 8, 4>(qd, qd, sd, sd, th, th, p2, u2, n2, s)
               : launch_q8<MODE_DOWN, 256, 6, 3, 8, 1>(qd, qd, sd, sd, th, thf2, p2, u2, n2, s);
}

}  // namespace moe
