// quant.cu -- Q8_0 block quantization of expert weights on the GPU (the
// prepare step of "Distributed MoE" (tenzro docs), quantization table:
// 32-element blocks with one f16 scale, about 8.5 bits per weight).
//
// For every block of 32 consecutive elements along K of a row:
//   amax = max |w|;  d = amax / 127;  id = d != 0 ? 1 / d : 0;
//   q = round-half-away(w * id);  scale = f16(d) (to nearest even)
// every step in IEEE fp32 with explicit rounding, so the integer codes are a
// deterministic function of the weights.  Codes keep the weight layout
// q[m][r][k]; scales are stored transposed per matrix, s[m][k/32][r], so a
// 128-row tile's scales for one 64-wide K block are two contiguous 256-byte
// runs (a TMA box).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const T* __restrict__ w, int n_mats,
                                                            int R, int K,
                                                            int8_t* __restrict__ q,
                                                            uint16_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long blk = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int nb = K / 32;
  if (blk >= (long long)n_mats * R * nb) return;
  const int b = (int)(blk % nb);
  const long long mr = blk / nb;  // m * R + r
  const int r = (int)(mr % R);
  const long long m = mr / R;
  const size_t i = (size_t)mr * K + (size_t)b * 32 + lane;
  const float v = load_as_f32(w, i);
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = __fdiv_rn(amax, 127.0f);
  const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
  q[i] = (int8_t)roundf(__fmul_rn(v, id));
  if (lane == 0)
    scales[((size_t)m * nb + b) * R + r] = __half_as_ushort(__float2half_rn(d));
}

}  // namespace

cudaError_t launch_quantize_q8_0(int dtype, const void* w, int n_mats, int R, int K, int8_t* q,
                                 uint16_t* scales, cudaStream_t s) {
  const long long blocks = (long long)n_mats * R * (K / 32);
  if (blocks == 0) return cudaSuccess;
  ProfScope pr("quantize_q8_0", s);
  const unsigned grid = (unsigned)((blocks + 7) / 8);
  if (dtype == MOE_BF16)
    (void)launch_kernel(quantize_q8_0_kernel<__nv_bfloat16>, grid, 256, 0, s,
                        static_cast<const __nv_bfloat16*>(w), n_mats, R, K, q, scales);
  else
    (void)launch_kernel(quantize_q8_0_kernel<float>, grid, 256, 0, s,
                        static_cast<const float*>(w), n_mats, R, K, q, scales);
  return cudaGetLastError();
}

}  // namespace moe
