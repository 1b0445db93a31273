// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/moe.h"

namespace moe {

// Workspace carve-up (every region 256-byte aligned).  Sizes follow the
// layer record; P = T * (k + S) is the number of (token, slot) pairs.
struct WsLayout {
  size_t flags;        // int32[4]: [0] error bits, [1] plan ticket
  size_t logits;       // fp32 [ksplit, T, E] partial router logits
  size_t topk_ids;     // int32 [T, k]
  size_t topk_w;       // fp32 [T, k]
  size_t offsets;      // int32 [E+S+1]
  size_t tok_idx;      // int32 [P]
  size_t slot_row;     // int32 [P]
  size_t active;       // int32 [E+S]
  size_t n_active;     // int32 [1]
  size_t slot_w;       // fp32 [P]
  size_t plan_bits;    // uint32 [E+S, ceil(T/32)]  token bitmap per expert
  size_t plan_wpre;    // int32 [E+S, ceil(T/32)]   popcount prefix per bitmap word
  size_t plan_counts;  // int32 [E+S]               batch sizes
  size_t x_perm;       // dtype [cap, d], cap = tc_row_capacity(P)
  size_t h;            // dtype [cap, I]
  size_t y_perm;       // dtype [P, d]
  size_t x_stage[2];   // dtype [T, d]: x of a call with host buffers (two: pipelined call)
  size_t y_stage[2];   // fp32 [T, d]:  y of a call with host buffers (two: pipelined call)
  size_t total;
};

WsLayout ws_layout(const moe_layer_desc& d);

// Rows of the permuted-row buffers for P batch rows (see tc_gemm.cu).
int tc_row_capacity(int P);

inline size_t dtype_size(int dt) { return dt == MOE_BF16 ? 2 : 4; }

// ---------------------------------------------------------------- profiling hooks
struct ProfScope {
  ProfScope(const char* name, cudaStream_t s, uint64_t bytes = 0);
  ~ProfScope();
  const char* name;
  cudaStream_t stream;
  int slot;
};
void count_launch();

// Launch with programmatic dependent launch allowed (see pdl_wait/pdl_trigger
// in common.cuh): the kernel may begin while its predecessor on the stream
// finishes.  Counts the launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.

// Router logits are produced as ksplit partial sums over K chunks,
// partial[chunk][T][E] fp32, summed in chunk order by the top-k kernel.
struct RouterPlan {
  int tc;      // 1: tcgen05 kernel (bf16, T >= 128, E >= 128); 0: CUDA-core split-K kernel
  int ksplit;  // number of K chunks (partial logit slices)
  int kb_per;  // tcgen05: 64-wide K blocks per chunk
  int kc;      // CUDA cores: elements per chunk
};
RouterPlan router_plan(int dtype, int T, int d, int E);

// CUDA cores: one warp per (expert, K chunk), router weights read once.
cudaError_t launch_router_logits_splitk(int dtype, const void* x, const void* Wr, int T, int d,
                                        int E, int kc, int ksplit, float* partial,
                                        cudaStream_t s);
// tcgen05 (bf16): 128 experts x 128 tokens x K chunk per unit.
cudaError_t launch_router_logits_tc(const void* x, const void* Wr, int T, int d, int E,
                                    int ksplit, int kb_per, float* partial, int* err,
                                    cudaStream_t s);
// One CTA waits on an mbarrier that nothing completes, with the bounded wait
// named by `which` (0 thread, 1 warp, 2 wind-down, 3 two waits sharing an
// abort flag); the wait expires and records kErrTimeout in *err.
cudaError_t launch_bounded_wait_check(int which, int* err, cudaStream_t s);
// per-token top-k and gate weights from the partial logits
cudaError_t launch_router_topk(const float* partial, int ksplit, const float* logit_bias,
                               const float* sel_bias, int T, int E, int k, int gate,
                               int norm_topk, float rs, int32_t* ids, float* w, cudaStream_t s);

cudaError_t launch_plan(const int32_t* ids, const float* topk_w, int T, int E, int k, int S,
                        int32_t* offsets, int32_t* tok_idx, int32_t* slot_row, int32_t* active,
                        int32_t* n_active, float* slot_w, uint32_t* bits, int32_t* wpre,
                        int32_t* counts, int* flags, cudaStream_t s);

// bf16 rows gathered into fp16 rows (operands of the Q8_0 GEMMs)
cudaError_t launch_gather_rows_to_f16(const void* x, const int32_t* tok_idx,
                                      const int32_t* total_rows, int P, int T, int d,
                                      void* x_perm, int* flags, cudaStream_t s);

// x_perm[slot_row[t, j]] = x[t] for every token t and slot j (dropped slots,
// -1, skipped); to_f16: bf16 rows written as fp16 rows
cudaError_t launch_scatter_rows(int dtype, bool to_f16, const void* x, const int32_t* slot_row,
                                const int32_t* total_rows, int T, int ks, int d, void* x_perm,
                                int* flags, cudaStream_t s);

// Expert loads of the host-memory tier (one launch, plain stream order): for
// each job (expert, slot), its three projections of mat_bytes each from
// host[0..2] (device-visible addresses of the host arrays) into pool[0..2].
constexpr int kMaxExpertLoadJobs = 1028;
struct ExpertLoadJobs {
  int2 job[kMaxExpertLoadJobs];  // x: expert, y: slot
};
cudaError_t launch_load_experts(const ExpertLoadJobs& jobs, int n, const void* const host[3],
                                void* const pool[3], size_t mat_bytes, cudaStream_t s);

cudaError_t launch_gather_rows(int dtype, const void* x, const int32_t* tok_idx,
                               const int32_t* total_rows, int P, int T, int d, void* x_perm,
                               int* flags, cudaStream_t s);

// fp32 SIMT expert FFN: h = silu(x_perm Wg^T) * (x_perm Wu^T); y_perm = (h Wd^T) * slot_w
cudaError_t launch_ffn_simt(const float* x_perm, const int32_t* offsets, int n_groups, int P,
                            int d, int I, const float* Wg, const float* Wu, const float* Wd,
                            const float* slot_w, float* h, float* y_perm, cudaStream_t s);

// bf16 tcgen05 expert FFN (gate/up + SwiGLU, then down).  With group_slot,
// group g's weights are matrix group_slot[g] of Wg/Wu/Wd, which then hold
// n_mats matrices (a slot pool); a negative entry skips the group's rows.
cudaError_t launch_ffn_tc(const void* x_perm, const int32_t* offsets, int n_groups, int P,
                          int d, int I, double mean_rows, const void* Wg, const void* Wu,
                          const void* Wd, const float* slot_w, void* h, void* y_perm, int* err,
                          cudaStream_t s, int n_mats = 0, const int32_t* group_slot = nullptr);

cudaError_t launch_combine(int dtype, const void* y_perm, const int32_t* slot_row,
                           const float* topk_w, const float* residual, int T, int d, int k,
                           int S, float* y, cudaStream_t s);

// Q8_0 expert weights: int8 codes [E+S, R, K] and f16 scales [E+S, K/32, R].
struct Q8Weight {
  const void* q;
  const void* scale;
};
cudaError_t launch_quantize_q8_0(int dtype, const void* w, int n_mats, int R, int K, int8_t* q,
                                 uint16_t* scales, cudaStream_t s);
cudaError_t launch_ffn_tc_q8(const void* x_perm, const int32_t* offsets, int n_groups, int P,
                             int d, int I, double mean_rows, const Q8Weight& Wg,
                             const Q8Weight& Wu, const Q8Weight& Wd, const float* slot_w,
                             void* h, void* y_perm, int* err, cudaStream_t s);

cudaError_t launch_combine_partial(int dtype, const void* y_perm, const int32_t* slot_row,
                                   const int32_t* ids, const float* topk_w,
                                   const int32_t* avail, const float* residual, int T, int d,
                                   int k, int S, int E, float* y, int32_t* missing,
                                   cudaStream_t s);

// (expert, token) of every slot flagged in missing [T, k+S], token-major
cudaError_t launch_missing_pairs(const int32_t* ids, const int32_t* missing, int T, int k,
                                 int S, int E, int32_t* pairs, int32_t* n_pairs,
                                 cudaStream_t s);

int num_sms();

// Expert residency in a bounded set of device slots (slot_cache.cu).
class SlotCache {
 public:
  SlotCache(int n_slots, int n_experts);
  // Slots for one step's distinct experts: slot[i], load[i] (1: its bytes
  // must be brought into the slot), pass[i] (passes run in order); false on a
  // bad argument (out of range or repeated expert), with nothing changed.
  bool assign(const int32_t* experts, int n, int32_t* slot, int32_t* load, int32_t* pass,
              int32_t* n_passes);
  int slot_of(int expert) const { return expert_slot_[expert]; }
  int n_slots() const { return (int)slot_expert_.size(); }
  int n_experts() const { return (int)expert_slot_.size(); }
  int resident() const;
  void fill_stats(moe_tier_stats* out) const;

 private:
  int pick() const;
  struct Counters {
    uint64_t steps = 0, hits = 0, misses = 0, evictions = 0, extra_passes = 0;
  };
  std::vector<int> slot_expert_, expert_slot_;
  std::vector<uint64_t> stamp_;  // step that last used the slot
  std::vector<char> pinned_;
  uint64_t clock_ = 0;
  Counters stats_;
};

}  // namespace moe
