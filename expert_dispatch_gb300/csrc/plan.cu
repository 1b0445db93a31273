// plan.cu -- the dispatch planner: routing (token -> experts) inverted into
// per-expert batches of token rows (expert -> tokens), as in the
// tenzro_moePlanDispatch records of "Distributed MoE" (tenzro docs): one
// batch of token_indices per (layer, expert), plus per-token slot
// assignments.
//
// The stable counting sort of the (token, slot) pairs in token-major order
// places a pair of token t in expert e's batch at rank #{t' < t : t' chose e},
// because a token chooses an expert at most once.  That rank is computed
// without any sequential pass:
//   1. plan_mark   : set bit t of expert e's token bitmap for every pair;
//   2. plan_scan   : per expert, an exclusive prefix of the bitmap words'
//                    popcounts and the batch size; the last block to finish
//                    turns the sizes into expert_offsets and the active list;
//   3. plan_place  : pos = offsets[e] + prefix(word) + popc(bits below t).
// Every result is a pure function of the routing (bit-reproducible).
#include "common.cuh"
#include "internal.h"
#include "route_plan.cuh"

namespace moe {
namespace {

__global__ void plan_mark(const int32_t* __restrict__ ids, int T, int E, int k, int S,
                          uint32_t* __restrict__ bits, int nw, int* __restrict__ flags) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  const long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int ks = k + S;
  if (p >= (long long)T * ks) return;
  const int t = (int)(p / ks), j = (int)(p % ks);
  const int e = rp::pair_expert(ids, t, j, k, E);
  if (j < k && (e < 0 || e >= E)) {
    flag_error(flags, kErrDeviceInput);
    return;
  }
  const uint32_t bit = 1u << (t & 31);
  const uint32_t old = atomicOr(&bits[(size_t)e * nw + (t >> 5)], bit);
  if (old & bit) flag_error(flags, kErrDeviceInput);  // an expert repeated within a token
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 256).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = lane < 8 ? warp_sums[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += u;
    }
    if (lane < 8) warp_sums[lane] = si - s;  // exclusive per-warp base
    if (lane == 7) *total = si;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();  // warp_sums may be reused by the caller
  return r;
}

// One block per expert: word prefixes of the token bitmap and the batch size.
// The last block to finish also turns batch sizes into offsets and the
// active-expert list.
__global__ void __launch_bounds__(256) plan_scan(const uint32_t* __restrict__ bits, int nw,
                                                 int nE, int32_t* __restrict__ wpre,
                                                 int32_t* __restrict__ counts,
                                                 int32_t* __restrict__ offsets,
                                                 int32_t* __restrict__ active,
                                                 int32_t* __restrict__ n_active,
                                                 int* __restrict__ ticket) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  __shared__ int warp_sums[8];
  __shared__ int chunk_total;
  __shared__ int is_last;
  const int e = blockIdx.x;
  int carry = 0;
  for (int w0 = 0; w0 < nw; w0 += 256) {
    const int w = w0 + threadIdx.x;
    const int c = w < nw ? __popc(bits[(size_t)e * nw + w]) : 0;
    const int ex = block_exclusive_scan(c, warp_sums, &chunk_total);
    if (w < nw) wpre[(size_t)e * nw + w] = carry + ex;
    __syncthreads();
    carry += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) counts[e] = carry;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // offsets = exclusive scan of counts; active = experts with count > 0
  int base = 0, abase = 0;
  for (int e0 = 0; e0 < nE; e0 += 256) {
    const int ee = e0 + threadIdx.x;
    const int c = ee < nE ? __ldcg(&counts[ee]) : 0;
    const int ex = block_exclusive_scan(c, warp_sums, &chunk_total);
    if (ee < nE) offsets[ee] = base + ex;
    __syncthreads();
    base += chunk_total;
    __syncthreads();
    const int a = (ee < nE && c > 0) ? 1 : 0;
    const int aex = block_exclusive_scan(a, warp_sums, &chunk_total);
    if (a && active) active[abase + aex] = ee;
    __syncthreads();
    abase += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    offsets[nE] = base;
    if (n_active) *n_active = abase;
    *ticket = 0;  // ready for the next call
  }
}

__global__ void plan_place(const int32_t* __restrict__ ids, const float* __restrict__ topk_w,
                           int T, int E, int k, int S, const uint32_t* __restrict__ bits, int nw,
                           const int32_t* __restrict__ wpre, const int32_t* __restrict__ offsets,
                           int32_t* __restrict__ tok_idx, int32_t* __restrict__ slot_row,
                           float* __restrict__ slot_w, int* __restrict__ flags) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  const long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int ks = k + S;
  const long long P = (long long)T * ks;
  if (p >= P) return;
  const int t = (int)(p / ks), j = (int)(p % ks);
  const int e = rp::pair_expert(ids, t, j, k, E);
  if (j < k && (e < 0 || e >= E)) {
    slot_row[p] = -1;
    return;
  }
  const size_t wi = (size_t)e * nw + (t >> 5);
  const uint32_t below = bits[wi] & ((1u << (t & 31)) - 1u);
  const long long pos = (long long)offsets[e] + wpre[wi] + __popc(below);
  if (pos < 0 || pos >= P) {  // offsets not made by this plan's scan: flagged, not written
    flag_error(flags, kErrDeviceInput);
    slot_row[p] = -1;
    return;
  }
  tok_idx[pos] = t;
  slot_row[p] = pos;
  if (slot_w) slot_w[pos] = (j < k && topk_w) ? topk_w[(size_t)t * k + j] : 1.f;
}

// The whole plan in one block (rp::plan_block), for problems whose token
// bitmaps fit in shared memory: the three steps above with the bitmaps, word
// prefixes and offsets kept on chip.  Same results, one launch.
constexpr int kSmallPlanThreads = 1024;
constexpr int kSmallPlanMaxWords = 4096;

__global__ void __launch_bounds__(kSmallPlanThreads) plan_small(
    const int32_t* __restrict__ ids, const float* __restrict__ topk_w, int T, int E, int k,
    int S, int nw, int32_t* __restrict__ offsets, int32_t* __restrict__ tok_idx,
    int32_t* __restrict__ slot_row, int32_t* __restrict__ active, int32_t* __restrict__ n_active,
    float* __restrict__ slot_w, int* __restrict__ flags) {
  pdl_wait();     // the predecessor grid is complete and visible
  pdl_trigger();  // dependents may launch (they wait for this grid in turn)
  extern __shared__ uint32_t sm[];
  __shared__ int warp_sums[32];
  __shared__ int chunk_total;
  rp::plan_block(ids, topk_w, T, E, k, S, nw, offsets, tok_idx, slot_row, active, n_active, slot_w,
                 flags, sm, warp_sums, &chunk_total);
}
}  // namespace

cudaError_t launch_plan(const int32_t* ids, const float* topk_w, int T, int E, int k, int S,
                        int32_t* offsets, int32_t* tok_idx, int32_t* slot_row, int32_t* active,
                        int32_t* n_active, float* slot_w, uint32_t* bits, int32_t* wpre,
                        int32_t* counts, int* flags, cudaStream_t s) {
  const int nE = E + S;
  const int nw = (T + 31) / 32;
  const long long P = (long long)T * (k + S);
  if ((long long)nE * nw <= kSmallPlanMaxWords && P <= 64ll * kSmallPlanThreads) {
    const size_t smem = sizeof(uint32_t) * (2 * (size_t)nE * nw + nE + 1);
    ProfScope pr("plan_small", s);
    (void)launch_kernel(plan_small, 1, kSmallPlanThreads, smem, s, ids, topk_w, T, E, k, S, nw, offsets, tok_idx,
                                                  slot_row, active, n_active, slot_w, flags);
    return cudaGetLastError();
  }
  cudaError_t err = cudaMemsetAsync(bits, 0, sizeof(uint32_t) * (size_t)nE * nw, s);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(flags + 1, 0, sizeof(int), s);  // ticket
  if (err != cudaSuccess) return err;
  const int nb = (int)((P + 255) / 256);
  {
    ProfScope pr("plan_mark", s);
    (void)launch_kernel(plan_mark, nb, 256, 0, s, ids, T, E, k, S, bits, nw, flags);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  {
    ProfScope pr("plan_scan", s);
    (void)launch_kernel(plan_scan, nE, 256, 0, s, bits, nw, nE, wpre, counts, offsets, active, n_active,
                                 flags + 1);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  {
    ProfScope pr("plan_place", s);
    (void)launch_kernel(plan_place, nb, 256, 0, s, ids, topk_w, T, E, k, S, bits, nw, wpre,
                        offsets, tok_idx, slot_row, slot_w, flags);
  }
  return cudaGetLastError();
}

}  // namespace moe
