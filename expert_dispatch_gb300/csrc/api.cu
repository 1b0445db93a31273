// api.cu -- the C ABI (include/moe.h): argument checks, workspace carve-up,
// and the stream-ordered launch sequences of the five layer calls.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

#include <nvtx3/nvToolsExt.h>

namespace moe {

namespace {

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A named NVTX range around each stream-ordered entry point, so a timeline
// profiler shows the library's calls (a no-op unless a tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

moe_status check_desc(const moe_layer_desc* D) {
  if (!D) return MOE_ERR_INVALID_ARG;
  if (D->T < 0 || D->d <= 0 || D->E <= 0 || D->E > 1024 || D->k <= 0 || D->k > D->E ||
      D->k > 32 || D->I <= 0 || D->S < 0 || D->S > 4)
    return MOE_ERR_INVALID_ARG;
  if (D->gate != MOE_GATE_SOFTMAX_TOPK && D->gate != MOE_GATE_SIGMOID_BIAS)
    return MOE_ERR_INVALID_ARG;
  if (D->norm_topk != 0 && D->norm_topk != 1) return MOE_ERR_INVALID_ARG;
  if (!isfinite(D->routed_scaling)) return MOE_ERR_INVALID_ARG;
  const long long P = (long long)D->T * (D->k + D->S);
  if (P > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
  if (D->dtype == MOE_BF16) {
    if (D->d % 64 || D->I % 64) return MOE_ERR_UNSUPPORTED;
    const long long ng = D->E + D->S;
    if (ng * D->I < 128 || ng * D->d < 128) return MOE_ERR_UNSUPPORTED;
  } else if (D->dtype == MOE_F32) {
    if (D->d % 8 || D->I % 4) return MOE_ERR_UNSUPPORTED;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

struct Ws {
  int* flags;
  float* logits;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* offsets;
  int32_t* tok_idx;
  int32_t* slot_row;
  int32_t* active;
  int32_t* n_active;
  float* slot_w;
  uint32_t* bits;
  int32_t* wpre;
  int32_t* counts;
  void* x_perm;
  void* h;
  void* y_perm;
  void* x_stage[2];
  float* y_stage[2];
};

Ws carve(void* base, const WsLayout& L) {
  uint8_t* b = static_cast<uint8_t*>(base);
  Ws w;
  w.flags = reinterpret_cast<int*>(b + L.flags);
  w.logits = reinterpret_cast<float*>(b + L.logits);
  w.topk_ids = reinterpret_cast<int32_t*>(b + L.topk_ids);
  w.topk_w = reinterpret_cast<float*>(b + L.topk_w);
  w.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  w.tok_idx = reinterpret_cast<int32_t*>(b + L.tok_idx);
  w.slot_row = reinterpret_cast<int32_t*>(b + L.slot_row);
  w.active = reinterpret_cast<int32_t*>(b + L.active);
  w.n_active = reinterpret_cast<int32_t*>(b + L.n_active);
  w.slot_w = reinterpret_cast<float*>(b + L.slot_w);
  w.bits = reinterpret_cast<uint32_t*>(b + L.plan_bits);
  w.wpre = reinterpret_cast<int32_t*>(b + L.plan_wpre);
  w.counts = reinterpret_cast<int32_t*>(b + L.plan_counts);
  w.x_perm = b + L.x_perm;
  w.h = b + L.h;
  w.y_perm = b + L.y_perm;
  for (int i = 0; i < 2; ++i) {
    w.x_stage[i] = b + L.x_stage[i];
    w.y_stage[i] = reinterpret_cast<float*>(b + L.y_stage[i]);
  }
  return w;
}

moe_status check_ws(const moe_layer_desc* D, void* ws, size_t bytes) {
  if (!ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  if (bytes < ws_layout(*D).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---------------------------------------------------------------- profiling
struct ProfRecord {
  std::string name;
  cudaEvent_t start, stop;
  uint64_t bytes;  // bytes the launch moves, when its launcher states them (else 0)
};
std::mutex g_prof_mu;
bool g_prof_on = false;
bool g_prof_bytes_only = false;  // record only launches that state the bytes they move
std::vector<ProfRecord> g_prof;
std::vector<cudaEvent_t> g_prof_free;
std::atomic<long long> g_launches{0};

cudaEvent_t take_event() {
  if (!g_prof_free.empty()) {
    cudaEvent_t e = g_prof_free.back();
    g_prof_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// The routing passes and the shared gating kernel.
// Routing and the dispatch plan of a layer call (no slot weights: the combine
// applies the gate weights).
moe_status do_route(const moe_layer_desc* D, const void* x, const void* Wr,
                    const float* logit_bias, const float* sel_bias, int32_t* ids, float* w,
                    const Ws& W, cudaStream_t s);
moe_status route_and_plan(const moe_layer_desc* D, const void* x, const void* Wr,
                          const float* logit_bias, const float* sel_bias, int32_t* ids, float* w,
                          const Ws& W, cudaStream_t s) {
  const moe_status st = do_route(D, x, Wr, logit_bias, sel_bias, ids, w, W, s);
  if (st != MOE_OK) return st;
  return cuda_status(launch_plan(ids, nullptr, D->T, D->E, D->k, D->S, W.offsets, W.tok_idx,
                                 W.slot_row, W.active, W.n_active, nullptr, W.bits, W.wpre,
                                 W.counts, W.flags, s));
}

moe_status do_route(const moe_layer_desc* D, const void* x, const void* Wr,
                    const float* logit_bias, const float* sel_bias, int32_t* ids, float* w,
                    const Ws& W, cudaStream_t s) {
  const RouterPlan rp = router_plan(D->dtype, D->T, D->d, D->E);
  const cudaError_t e =
      rp.tc ? launch_router_logits_tc(x, Wr, D->T, D->d, D->E, rp.ksplit, rp.kb_per, W.logits,
                                      W.flags, s)
            : launch_router_logits_splitk(D->dtype, x, Wr, D->T, D->d, D->E, rp.kc, rp.ksplit,
                                          W.logits, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_router_topk(W.logits, rp.ksplit, logit_bias, sel_bias, D->T, D->E,
                                        D->k, D->gate, D->norm_topk, D->routed_scaling, ids, w,
                                        s));
}

// Batch rows are permuted into x_perm from the token side when the plan's
// slot_row map is at hand (the layer call), else from the row side.
cudaError_t permute_rows(const moe_layer_desc* D, bool to_f16, const void* x,
                         const int32_t* offsets, const int32_t* tok_idx, const int32_t* slot_row,
                         const Ws& W, cudaStream_t s) {
  const int P = D->T * (D->k + D->S);
  const int nE = D->E + D->S;
  if (slot_row)
    return launch_scatter_rows(D->dtype, to_f16, x, slot_row, offsets + nE, D->T, D->k + D->S,
                               D->d, W.x_perm, W.flags, s);
  return to_f16 ? launch_gather_rows_to_f16(x, tok_idx, offsets + nE, P, D->T, D->d, W.x_perm,
                                            W.flags, s)
                : launch_gather_rows(D->dtype, x, tok_idx, offsets + nE, P, D->T, D->d,
                                     W.x_perm, W.flags, s);
}

moe_status do_ffn(const moe_layer_desc* D, const void* x, const int32_t* offsets,
                  const int32_t* tok_idx, const int32_t* slot_row, const float* slot_w,
                  const void* Wg, const void* Wu, const void* Wd, void* y_perm, const Ws& W,
                  cudaStream_t s) {
  const int P = D->T * (D->k + D->S);
  const int nE = D->E + D->S;
  cudaError_t e = permute_rows(D, false, x, offsets, tok_idx, slot_row, W, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (D->dtype == MOE_F32) {
    e = launch_ffn_simt(static_cast<const float*>(W.x_perm), offsets, nE, P, D->d, D->I,
                        static_cast<const float*>(Wg), static_cast<const float*>(Wu),
                        static_cast<const float*>(Wd), slot_w, static_cast<float*>(W.h),
                        static_cast<float*>(y_perm), s);
  } else {
    const double mean_rows = (double)P / (double)nE;
    e = launch_ffn_tc(W.x_perm, offsets, nE, P, D->d, D->I, mean_rows, Wg, Wu, Wd, slot_w, W.h,
                      y_perm, W.flags, s);
  }
  return cuda_status(e);
}

// The same with Q8_0 expert weights (bf16 activations).
moe_status do_ffn_q8(const moe_layer_desc* D, const void* x, const int32_t* offsets,
                     const int32_t* tok_idx, const int32_t* slot_row, const float* slot_w,
                     const moe_q8_weight* Wg, const moe_q8_weight* Wu, const moe_q8_weight* Wd,
                     void* y_perm, const Ws& W, cudaStream_t s) {
  const int P = D->T * (D->k + D->S);
  const int nE = D->E + D->S;
  if (permute_rows(D, true, x, offsets, tok_idx, slot_row, W, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  const Q8Weight g{Wg->q, Wg->scale}, u{Wu->q, Wu->scale}, dn{Wd->q, Wd->scale};
  return cuda_status(launch_ffn_tc_q8(W.x_perm, offsets, nE, P, D->d, D->I, (double)P / nE, g, u,
                                      dn, slot_w, W.h, y_perm, W.flags, s));
}

bool q8_ok(const moe_q8_weight* w) {
  return w && w->q && w->scale && aligned16(w->q) && aligned16(w->scale);
}

}  // namespace

RouterPlan router_plan(int dtype, int T, int d, int E) {
  RouterPlan r{};
  if (dtype == MOE_BF16 && T >= 32 && E >= 128) {
    // enough units (128 experts x 128 tokens x K chunk) for ~2 per SM, at most 16 chunks
    r.tc = 1;
    const int KB = d / 64;
    const int base = ((E + 127) / 128) * ((T + 127) / 128);
    int ks = (296 + base - 1) / base;
    ks = ks < 1 ? 1 : ks;
    ks = ks > 16 ? 16 : ks;
    ks = ks > KB ? KB : ks;
    r.kb_per = (KB + ks - 1) / ks;
    r.ksplit = (KB + r.kb_per - 1) / r.kb_per;
  } else {
    // one block per expert row keeps up to 4 x 256 16-byte vectors in registers
    r.kc = dtype == MOE_BF16 ? 8192 : 4096;
    r.ksplit = (d + r.kc - 1) / r.kc;
  }
  return r;
}

WsLayout ws_layout(const moe_layer_desc& D) {
  WsLayout L{};
  const size_t T = (size_t)D.T, E = (size_t)D.E, k = (size_t)D.k, S = (size_t)D.S;
  const size_t nE = E + S, P = T * (k + S);
  const size_t nw = (T + 31) / 32;
  const size_t cap = (size_t)tc_row_capacity((int)P);
  const size_t es = dtype_size(D.dtype);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.flags = take(16);
  L.logits = take((size_t)router_plan(D.dtype, D.T, D.d, D.E).ksplit * T * E * 4);
  L.topk_ids = take(T * k * 4);
  L.topk_w = take(T * k * 4);
  L.offsets = take((nE + 1) * 4);
  L.tok_idx = take(P * 4);
  L.slot_row = take(P * 4);
  L.active = take(nE * 4);
  L.n_active = take(4);
  L.slot_w = take(P * 4);
  L.plan_bits = take(nE * nw * 4);
  L.plan_wpre = take(nE * nw * 4);
  L.plan_counts = take(nE * 4);
  L.x_perm = take(cap * (size_t)D.d * es);
  L.h = take(cap * (size_t)D.I * es);
  L.y_perm = take(P * (size_t)D.d * es);
  for (int i = 0; i < 2; ++i) {
    L.x_stage[i] = take(T * (size_t)D.d * es);
    L.y_stage[i] = take(T * (size_t)D.d * 4);
  }
  L.total = off;
  return L;
}

ProfScope::ProfScope(const char* n, cudaStream_t s, uint64_t bytes)
    : name(n), stream(s), slot(-1) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  if (!g_prof_on || (g_prof_bytes_only && bytes == 0)) return;
  ProfRecord r{n, take_event(), take_event(), bytes};
  if (!r.start || !r.stop) return;
  if (cudaEventRecord(r.start, s) != cudaSuccess) return;
  g_prof.push_back(r);
  slot = (int)g_prof.size() - 1;
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> g(g_prof_mu);
  if (slot < (int)g_prof.size()) cudaEventRecord(g_prof[slot].stop, stream);
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace moe

using namespace moe;

// The expert tier: host-resident expert projections, a pool of HBM slots and
// the slot cache deciding residency (slot_cache.cu).
struct moe_expert_tier {
  moe_layer_desc desc{};
  int device = 0;
  int nE = 0, n_slots = 0;
  size_t mat_bytes = 0;  // one expert's Wg (= Wu = Wd) bytes
  const uint8_t* host[3] = {nullptr, nullptr, nullptr};
  const void* host_dev[3] = {nullptr, nullptr, nullptr};  // device-visible addresses, or null
  bool registered[3] = {false, false, false};
  void* pool[3] = {nullptr, nullptr, nullptr};  // Wg, Wu, Wd slots
  int32_t* host_tab = nullptr;  // pinned: [nE + 1] batch bounds, then [nE][nE] pass tables
  int32_t* dev_tab = nullptr;   // [nE][nE] pass tables
  cudaEvent_t done = nullptr;
  bool done_recorded = false;
  // Slot loads run on a stream of their own, joined to the caller's by
  // events: large host -> device copies enqueued between kernels launched
  // with programmatic dependent launch ran at a fraction of the link's
  // bandwidth, and a load kernel there would be the programmatic predecessor
  // of the FFN kernel that reads what it wrote.
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ready = nullptr, copied = nullptr;
  uint64_t bytes_loaded = 0;
  SlotCache cache;
  std::mutex mu;
  moe_expert_tier(int slots, int experts) : cache(slots, experts) {}
};

namespace {

void tier_free(moe_expert_tier* t) {
  if (!t) return;
  if (t->done) {
    if (t->done_recorded) cudaEventSynchronize(t->done);
    cudaEventDestroy(t->done);
  }
  for (int i = 0; i < 3; ++i) {
    if (t->pool[i]) cudaFree(t->pool[i]);
    if (t->registered[i]) cudaHostUnregister(const_cast<uint8_t*>(t->host[i]));
  }
  if (t->dev_tab) cudaFree(t->dev_tab);
  if (t->host_tab) cudaFreeHost(t->host_tab);
  if (t->copy_stream) {
    cudaStreamSynchronize(t->copy_stream);
    cudaStreamDestroy(t->copy_stream);
  }
  if (t->ready) cudaEventDestroy(t->ready);
  if (t->copied) cudaEventDestroy(t->copied);
  delete t;
}

// Copy expert e's three projections into `slot` (host -> device, on stream s).
moe_status tier_load(moe_expert_tier* t, int e, int slot, cudaStream_t s);

// Load the listed experts (load[i] set, of pass p unless pass is null) into
// their slots on the tier's copy stream, after everything enqueued on s so far
// (so no slot is overwritten while earlier kernels read it); work enqueued on
// s afterwards waits for them.  One load kernel when the host arrays are
// device-visible, else three copies per expert.
moe_status tier_load_all(moe_expert_tier* t, const int32_t* experts, const int32_t* slot,
                         const int32_t* load, const int32_t* pass, int n, int p,
                         cudaStream_t s) {
  ExpertLoadJobs jobs;
  int n_jobs = 0;
  for (int i = 0; i < n; ++i) {
    if (!load[i] || (pass != nullptr && pass[i] != p)) continue;
    if (experts[i] < 0 || experts[i] >= t->nE || slot[i] < 0 || slot[i] >= t->n_slots ||
        n_jobs >= kMaxExpertLoadJobs)
      return MOE_ERR_INVALID_ARG;
    jobs.job[n_jobs++] = make_int2(experts[i], slot[i]);
  }
  if (n_jobs == 0) return MOE_OK;
  if (cudaEventRecord(t->ready, s) != cudaSuccess ||
      cudaStreamWaitEvent(t->copy_stream, t->ready, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (t->host_dev[0] && t->host_dev[1] && t->host_dev[2]) {
    if (launch_load_experts(jobs, n_jobs, t->host_dev, t->pool, t->mat_bytes, t->copy_stream) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    t->bytes_loaded += (uint64_t)n_jobs * 3 * t->mat_bytes;
  } else {
    for (int j = 0; j < n_jobs; ++j) {
      const moe_status st = tier_load(t, jobs.job[j].x, jobs.job[j].y, t->copy_stream);
      if (st != MOE_OK) return st;
    }
  }
  if (cudaEventRecord(t->copied, t->copy_stream) != cudaSuccess ||
      cudaStreamWaitEvent(s, t->copied, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status tier_load(moe_expert_tier* t, int e, int slot, cudaStream_t s) {
  for (int i = 0; i < 3; ++i) {
    if (cudaMemcpyAsync(static_cast<uint8_t*>(t->pool[i]) + (size_t)slot * t->mat_bytes,
                        t->host[i] + (size_t)e * t->mat_bytes, t->mat_bytes,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  t->bytes_loaded += 3 * t->mat_bytes;
  return MOE_OK;
}


// A run of layer calls on host buffers with the copies off the compute stream.
// Step i computes from x stage i % 2 into y stage i % 2 on `stream`; an upload
// stream brings x_host[i + 1] into the other x stage while step i computes, and
// a download stream takes y stage i to y_host[i] while step i + 1 computes.
// Events order the three streams:
//   upload i + 1   after  step i - 1 (its x stage was read there)
//   step i         after  upload i, and after download i - 2 (its y stage)
//   download i     after  step i
// The run begins after the work on `stream` before the call (both copy
// streams wait for it) and `stream` waits for the last download, so work
// enqueued after the call sees every y_host[i] written.  The copy streams and
// events are the call's own and are released once their work completes.
struct PipelineRes {
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, x_ready[2] = {}, computed[2] = {}, y_done[2] = {};
  ~PipelineRes() {
    cudaEvent_t* evs[] = {&start, &x_ready[0], &x_ready[1], &computed[0], &computed[1],
                          &y_done[0], &y_done[1]};
    for (cudaEvent_t* e : evs)
      if (*e) cudaEventDestroy(*e);
    if (up) cudaStreamDestroy(up);
    if (down) cudaStreamDestroy(down);
  }
  bool create() {
    if (cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking) != cudaSuccess)
      return false;
    cudaEvent_t* evs[] = {&start, &x_ready[0], &x_ready[1], &computed[0], &computed[1],
                          &y_done[0], &y_done[1]};
    for (cudaEvent_t* e : evs)
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
};

template <typename LayerFn>
moe_status forward_host_pipelined(const moe_layer_desc* desc, int n_steps,
                                  const void* const* x_host, float* const* y_host,
                                  void* workspace, size_t ws_bytes, void* stream,
                                  const LayerFn& layer) {
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (n_steps < 0) return MOE_ERR_INVALID_ARG;
  if (n_steps == 0 || desc->T == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_steps; ++i)
    if (!x_host[i] || !y_host[i]) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  const Ws W = carve(workspace, ws_layout(*desc));
  const size_t xb = (size_t)desc->T * desc->d * dtype_size(desc->dtype);
  const size_t yb = (size_t)desc->T * desc->d * 4;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PipelineRes R;
  if (!R.create()) return MOE_ERR_CUDA;
  bool ok = cudaEventRecord(R.start, s) == cudaSuccess &&
            cudaStreamWaitEvent(R.up, R.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(R.down, R.start, 0) == cudaSuccess;
  auto upload = [&](int i) {
    const int b = i & 1;
    return (i < 2 || cudaStreamWaitEvent(R.up, R.computed[b], 0) == cudaSuccess) &&
           cudaMemcpyAsync(W.x_stage[b], x_host[i], xb, cudaMemcpyHostToDevice, R.up) ==
               cudaSuccess &&
           cudaEventRecord(R.x_ready[b], R.up) == cudaSuccess;
  };
  ok = ok && upload(0);
  for (int i = 0; ok && i < n_steps; ++i) {
    const int b = i & 1;
    if (i + 1 < n_steps && !(ok = upload(i + 1))) break;
    if (cudaStreamWaitEvent(s, R.x_ready[b], 0) != cudaSuccess ||
        (i >= 2 && cudaStreamWaitEvent(s, R.y_done[b], 0) != cudaSuccess)) {
      ok = false;
      break;
    }
    if ((st = layer(W.x_stage[b], W.y_stage[b])) != MOE_OK) break;
    ok = cudaEventRecord(R.computed[b], s) == cudaSuccess &&
         cudaStreamWaitEvent(R.down, R.computed[b], 0) == cudaSuccess &&
         cudaMemcpyAsync(y_host[i], W.y_stage[b], yb, cudaMemcpyDeviceToHost, R.down) ==
             cudaSuccess &&
         cudaEventRecord(R.y_done[b], R.down) == cudaSuccess;
  }
  // join: whatever was enqueued on the copy streams ends before later work on `stream`
  const bool joined = cudaEventRecord(R.x_ready[0], R.up) == cudaSuccess &&
                      cudaEventRecord(R.y_done[0], R.down) == cudaSuccess &&
                      cudaStreamWaitEvent(s, R.x_ready[0], 0) == cudaSuccess &&
                      cudaStreamWaitEvent(s, R.y_done[0], 0) == cudaSuccess;
  if (st != MOE_OK) return st;
  return ok && joined ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

moe_status moe_workspace_size(const moe_layer_desc* desc, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  *bytes = desc->T == 0 ? 0 : ws_layout(*desc).total;
  return MOE_OK;
}

moe_status moe_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || ws_bytes < 16 || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, 16, static_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const moe_layer_desc* desc, const void* x, const void* Wr,
                     const float* logit_bias, const float* sel_bias, int32_t* topk_ids,
                     float* topk_w, void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_route");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->T == 0) return MOE_OK;
  if (!x || !Wr || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(topk_ids) || !aligned16(topk_w))
    return MOE_ERR_INVALID_ARG;
  if (sel_bias && desc->gate != MOE_GATE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  const Ws W = carve(workspace, ws_layout(*desc));
  return do_route(desc, x, Wr, logit_bias, sel_bias, topk_ids, topk_w, W,
                  static_cast<cudaStream_t>(stream));
}

moe_status moe_plan_dispatch(const moe_layer_desc* desc, const int32_t* topk_ids,
                             const float* topk_w, int32_t* expert_offsets,
                             int32_t* token_indices, int32_t* slot_row, int32_t* active_ids,
                             int32_t* n_active, float* slot_w, void* workspace, size_t ws_bytes,
                             void* stream) {
  const NvtxRange nvtx("moe_plan_dispatch");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->T == 0) return MOE_OK;
  if (!topk_ids || !expert_offsets || !token_indices || !slot_row) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  const Ws W = carve(workspace, ws_layout(*desc));
  return cuda_status(launch_plan(topk_ids, topk_w, desc->T, desc->E, desc->k, desc->S,
                                 expert_offsets, token_indices, slot_row, active_ids, n_active,
                                 slot_w, W.bits, W.wpre, W.counts, W.flags,
                                 static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn(const moe_layer_desc* desc, const void* x,
                          const int32_t* expert_offsets, const int32_t* token_indices,
                          const float* slot_w, const void* Wg, const void* Wu, const void* Wd,
                          void* y_perm, void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_expert_ffn");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->T == 0) return MOE_OK;
  if (!x || !expert_offsets || !token_indices || !Wg || !Wu || !Wd || !y_perm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  const Ws W = carve(workspace, ws_layout(*desc));
  return do_ffn(desc, x, expert_offsets, token_indices, nullptr, slot_w, Wg, Wu, Wd, y_perm,
                W, static_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_layer_desc* desc, const void* y_perm, const int32_t* slot_row,
                       const float* topk_w, const float* residual, float* y, void* stream) {
  const NvtxRange nvtx("moe_combine");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->T == 0) return MOE_OK;
  if (!y_perm || !slot_row || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(desc->dtype, y_perm, slot_row, topk_w, residual, desc->T,
                                    desc->d, desc->k, desc->S, y,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_q8_0(int n_mats, int rows, int K, int src_dtype, const void* w, void* q,
                             void* scale, void* stream) {
  const NvtxRange nvtx("moe_quantize_q8_0");
  if (n_mats < 0 || rows <= 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
  if (src_dtype != MOE_F32 && src_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (n_mats == 0) return MOE_OK;
  if (!w || !q || !scale) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_q8_0(src_dtype, w, n_mats, rows, K,
                                          static_cast<int8_t*>(q), static_cast<uint16_t*>(scale),
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn_q8(const moe_layer_desc* desc, const void* x,
                             const int32_t* expert_offsets, const int32_t* token_indices,
                             const float* slot_w, const moe_q8_weight* Wg,
                             const moe_q8_weight* Wu, const moe_q8_weight* Wd, void* y_perm,
                             void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_expert_ffn_q8");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (desc->T == 0) return MOE_OK;
  if (!x || !expert_offsets || !token_indices || !y_perm || !q8_ok(Wg) || !q8_ok(Wu) ||
      !q8_ok(Wd) || !aligned16(x) || !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  const Ws W = carve(workspace, ws_layout(*desc));
  return do_ffn_q8(desc, x, expert_offsets, token_indices, nullptr, slot_w, Wg, Wu, Wd, y_perm,
                   W, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward_q8(const moe_layer_desc* desc, const void* x, const void* Wr,
                                const float* logit_bias, const float* sel_bias,
                                const moe_q8_weight* Wg, const moe_q8_weight* Wu,
                                const moe_q8_weight* Wd, const float* residual, float* y,
                                int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                                size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_layer_forward_q8");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (desc->T == 0) return MOE_OK;
  if (!x || !Wr || !y || !q8_ok(Wg) || !q8_ok(Wu) || !q8_ok(Wd)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(y) || (residual && !aligned16(residual)) ||
      (topk_ids_out && !aligned16(topk_ids_out)) || (topk_w_out && !aligned16(topk_w_out)))
    return MOE_ERR_INVALID_ARG;
  if (sel_bias && desc->gate != MOE_GATE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Ws W = carve(workspace, ws_layout(*desc));
  int32_t* ids = topk_ids_out ? topk_ids_out : W.topk_ids;
  float* w = topk_w_out ? topk_w_out : W.topk_w;
  if (cudaMemsetAsync(W.flags, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = route_and_plan(desc, x, Wr, logit_bias, sel_bias, ids, w, W, s)) != MOE_OK) return st;
  if ((st = do_ffn_q8(desc, x, W.offsets, W.tok_idx, W.slot_row, nullptr, Wg, Wu, Wd, W.y_perm,
                      W, s)) !=
      MOE_OK)
    return st;
  return cuda_status(launch_combine(desc->dtype, W.y_perm, W.slot_row, w, residual, desc->T,
                                    desc->d, desc->k, desc->S, y, s));
}

// The layer call with host buffers: x_host -> the workspace's x rows, the
// layer on the device, its y rows -> y_host; all on `stream`.
static moe_status forward_host_common(const moe_layer_desc* desc, const void* x_host,
                                      float* y_host, void* workspace, size_t ws_bytes,
                                      void* stream, const void** x_dev, float** y_dev) {
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  const Ws W = carve(workspace, ws_layout(*desc));
  *x_dev = W.x_stage[0];
  *y_dev = W.y_stage[0];
  const size_t bytes = (size_t)desc->T * desc->d * dtype_size(desc->dtype);
  return cuda_status(cudaMemcpyAsync(W.x_stage[0], x_host, bytes, cudaMemcpyHostToDevice,
                                     static_cast<cudaStream_t>(stream)));
}

static moe_status copy_y_to_host(const moe_layer_desc* desc, const float* y_dev, float* y_host,
                                 void* stream) {
  return cuda_status(cudaMemcpyAsync(y_host, y_dev, (size_t)desc->T * desc->d * 4,
                                     cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream)));
}

moe_status moe_layer_forward_host(const moe_layer_desc* desc, const void* x_host,
                                  const void* Wr, const float* logit_bias,
                                  const float* sel_bias, const void* Wg, const void* Wu,
                                  const void* Wd, const float* residual, float* y_host,
                                  int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                                  size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_layer_forward_host");
  if (desc && desc->T == 0 && check_desc(desc) == MOE_OK) return MOE_OK;
  const void* x = nullptr;
  float* y = nullptr;
  moe_status st = forward_host_common(desc, x_host, y_host, workspace, ws_bytes, stream, &x, &y);
  if (st != MOE_OK) return st;
  if ((st = moe_layer_forward(desc, x, Wr, logit_bias, sel_bias, Wg, Wu, Wd, residual, y,
                              topk_ids_out, topk_w_out, workspace, ws_bytes, stream)) != MOE_OK)
    return st;
  return copy_y_to_host(desc, y, y_host, stream);
}

moe_status moe_layer_forward_q8_host(const moe_layer_desc* desc, const void* x_host,
                                     const void* Wr, const float* logit_bias,
                                     const float* sel_bias, const moe_q8_weight* Wg,
                                     const moe_q8_weight* Wu, const moe_q8_weight* Wd,
                                     const float* residual, float* y_host,
                                     int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                                     size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_layer_forward_q8_host");
  if (desc && desc->T == 0 && check_desc(desc) == MOE_OK) return MOE_OK;
  const void* x = nullptr;
  float* y = nullptr;
  moe_status st = forward_host_common(desc, x_host, y_host, workspace, ws_bytes, stream, &x, &y);
  if (st != MOE_OK) return st;
  if ((st = moe_layer_forward_q8(desc, x, Wr, logit_bias, sel_bias, Wg, Wu, Wd, residual, y,
                                 topk_ids_out, topk_w_out, workspace, ws_bytes, stream)) !=
      MOE_OK)
    return st;
  return copy_y_to_host(desc, y, y_host, stream);
}

moe_status moe_layer_forward_host_pipelined(const moe_layer_desc* desc, int n_steps,
                                            const void* const* x_host, const void* Wr,
                                            const float* logit_bias, const float* sel_bias,
                                            const void* Wg, const void* Wu, const void* Wd,
                                            float* const* y_host, void* workspace,
                                            size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_layer_forward_host_pipelined");
  return forward_host_pipelined(
      desc, n_steps, x_host, y_host, workspace, ws_bytes, stream,
      [&](const void* x, float* y) {
        return moe_layer_forward(desc, x, Wr, logit_bias, sel_bias, Wg, Wu, Wd, nullptr, y,
                                 nullptr, nullptr, workspace, ws_bytes, stream);
      });
}

moe_status moe_layer_forward_q8_host_pipelined(const moe_layer_desc* desc, int n_steps,
                                               const void* const* x_host, const void* Wr,
                                               const float* logit_bias, const float* sel_bias,
                                               const moe_q8_weight* Wg, const moe_q8_weight* Wu,
                                               const moe_q8_weight* Wd, float* const* y_host,
                                               void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_layer_forward_q8_host_pipelined");
  return forward_host_pipelined(
      desc, n_steps, x_host, y_host, workspace, ws_bytes, stream,
      [&](const void* x, float* y) {
        return moe_layer_forward_q8(desc, x, Wr, logit_bias, sel_bias, Wg, Wu, Wd, nullptr, y,
                                    nullptr, nullptr, workspace, ws_bytes, stream);
      });
}

moe_status moe_combine_partial(const moe_layer_desc* desc, const void* y_perm,
                               const int32_t* slot_row, const int32_t* topk_ids,
                               const float* topk_w, const int32_t* expert_available,
                               const float* residual, float* y, int32_t* missing,
                               void* stream) {
  const NvtxRange nvtx("moe_combine_partial");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->T == 0) return MOE_OK;
  if (!y_perm || !slot_row || !topk_ids || !topk_w || !expert_available || !y)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine_partial(desc->dtype, y_perm, slot_row, topk_ids, topk_w,
                                            expert_available, residual, desc->T, desc->d,
                                            desc->k, desc->S, desc->E, y, missing,
                                            static_cast<cudaStream_t>(stream)));
}

moe_status moe_partial_missing_pairs(const moe_layer_desc* desc, const int32_t* topk_ids,
                                    const int32_t* missing, int32_t* pairs, int32_t* n_pairs,
                                    void* stream) {
  const NvtxRange nvtx("moe_partial_missing_pairs");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (!n_pairs) return MOE_ERR_INVALID_ARG;
  if (desc->T > 0 && (!topk_ids || !missing || !pairs)) return MOE_ERR_INVALID_ARG;
  if (pairs && (reinterpret_cast<uintptr_t>(pairs) & 7u)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_missing_pairs(topk_ids, missing, desc->T, desc->k, desc->S, desc->E,
                                          pairs, n_pairs, static_cast<cudaStream_t>(stream)));
}

moe_status moe_layer_forward(const moe_layer_desc* desc, const void* x, const void* Wr,
                             const float* logit_bias, const float* sel_bias, const void* Wg,
                             const void* Wu, const void* Wd, const float* residual, float* y,
                             int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                             size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_layer_forward");
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->T == 0) return MOE_OK;
  if (!x || !Wr || !Wg || !Wu || !Wd || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) ||
      !aligned16(y) || (residual && !aligned16(residual)) ||
      (topk_ids_out && !aligned16(topk_ids_out)) || (topk_w_out && !aligned16(topk_w_out)))
    return MOE_ERR_INVALID_ARG;
  if (sel_bias && desc->gate != MOE_GATE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Ws W = carve(workspace, ws_layout(*desc));
  int32_t* ids = topk_ids_out ? topk_ids_out : W.topk_ids;
  float* w = topk_w_out ? topk_w_out : W.topk_w;
  if (cudaMemsetAsync(W.flags, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = route_and_plan(desc, x, Wr, logit_bias, sel_bias, ids, w, W, s)) != MOE_OK) return st;
  if ((st = do_ffn(desc, x, W.offsets, W.tok_idx, W.slot_row, nullptr, Wg, Wu, Wd, W.y_perm, W,
                   s)) != MOE_OK)
    return st;
  return cuda_status(launch_combine(desc->dtype, W.y_perm, W.slot_row, w, residual, desc->T,
                                    desc->d, desc->k, desc->S, y, s));
}

moe_status moe_tier_create(const moe_layer_desc* desc, const void* Wg_host, const void* Wu_host,
                           const void* Wd_host, size_t hbm_budget_bytes, moe_expert_tier** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_layer_desc D = desc ? *desc : moe_layer_desc{};
  D.T = 1;  // the tier's shape check does not depend on T
  moe_status st = check_desc(desc ? &D : nullptr);
  if (st != MOE_OK) return st;
  if (D.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (!Wg_host || !Wu_host || !Wd_host) return MOE_ERR_INVALID_ARG;
  const int nE = D.E + D.S;
  const size_t mat_bytes = (size_t)D.I * D.d * 2;
  const size_t slots = hbm_budget_bytes / (3 * mat_bytes);
  if (slots < 1) return MOE_ERR_INVALID_ARG;
  const int n_slots = slots > (size_t)nE ? nE : (int)slots;
  moe_expert_tier* t = new moe_expert_tier(n_slots, nE);
  t->desc = D;
  t->nE = nE;
  t->n_slots = n_slots;
  t->mat_bytes = mat_bytes;
  t->host[0] = static_cast<const uint8_t*>(Wg_host);
  t->host[1] = static_cast<const uint8_t*>(Wu_host);
  t->host[2] = static_cast<const uint8_t*>(Wd_host);
  if (cudaGetDevice(&t->device) != cudaSuccess) {
    tier_free(t);
    return MOE_ERR_CUDA;
  }
  for (int i = 0; i < 3; ++i) {
    // page-lock the host copy so that slot loads are asynchronous DMA; memory
    // that is already page-locked is used as it is
    const cudaError_t e = cudaHostRegister(const_cast<uint8_t*>(t->host[i]),
                                           (size_t)nE * mat_bytes, cudaHostRegisterDefault);
    if (e == cudaSuccess)
      t->registered[i] = true;
    else
      (void)cudaGetLastError();
    // the device-visible address of page-locked, mapped host memory (null
    // when there is none: slot loads then use copies)
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, const_cast<uint8_t*>(t->host[i]), 0) == cudaSuccess &&
        (reinterpret_cast<uintptr_t>(dp) & 15u) == 0)
      t->host_dev[i] = dp;
    else
      (void)cudaGetLastError();
    if (cudaMalloc(&t->pool[i], (size_t)n_slots * mat_bytes) != cudaSuccess) {
      (void)cudaGetLastError();
      tier_free(t);
      return MOE_ERR_CUDA;
    }
  }
  if (cudaHostAlloc(reinterpret_cast<void**>(&t->host_tab),
                    ((size_t)nE + 1 + (size_t)nE * nE) * 4, cudaHostAllocDefault) !=
          cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&t->dev_tab), (size_t)nE * nE * 4) != cudaSuccess ||
      cudaEventCreateWithFlags(&t->done, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&t->ready, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&t->copied, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&t->copy_stream, cudaStreamNonBlocking) != cudaSuccess) {
    (void)cudaGetLastError();
    tier_free(t);
    return MOE_ERR_CUDA;
  }
  *out = t;
  return MOE_OK;
}

moe_status moe_tier_destroy(moe_expert_tier* tier) {
  tier_free(tier);
  return MOE_OK;
}

moe_status moe_tier_get_stats(moe_expert_tier* tier, moe_tier_stats* out) {
  if (!tier || !out) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(tier->mu);
  tier->cache.fill_stats(out);
  out->bytes_loaded = tier->bytes_loaded;
  return MOE_OK;
}

moe_status moe_tier_prefetch(moe_expert_tier* tier, const int32_t* experts, int n, void* stream) {
  const NvtxRange nvtx("moe_tier_prefetch");
  if (!tier || n < 0 || (n > 0 && !experts)) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(tier->mu);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n > tier->n_slots) n = tier->n_slots;  // the rest could not stay resident anyway
  if (n == 0) return MOE_OK;
  std::vector<int32_t> slot(n), load(n), pass(n);
  int32_t n_passes = 0;
  if (!tier->cache.assign(experts, n, slot.data(), load.data(), pass.data(), &n_passes))
    return MOE_ERR_INVALID_ARG;
  if (tier->done_recorded && cudaStreamWaitEvent(s, tier->done, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  const moe_status st =
      tier_load_all(tier, experts, slot.data(), load.data(), nullptr, n, 0, s);
  if (st != MOE_OK) return st;
  if (cudaEventRecord(tier->done, s) != cudaSuccess) return MOE_ERR_CUDA;
  tier->done_recorded = true;
  return MOE_OK;
}

moe_status moe_tier_forward(moe_expert_tier* tier, const moe_layer_desc* desc, const void* x,
                            const void* Wr, const float* logit_bias, const float* sel_bias,
                            const float* residual, float* y, int32_t* topk_ids_out,
                            float* topk_w_out, void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("moe_tier_forward");
  if (!tier) return MOE_ERR_INVALID_ARG;
  moe_status st = check_desc(desc);
  if (st != MOE_OK) return st;
  const moe_layer_desc& T0 = tier->desc;
  if (desc->d != T0.d || desc->E != T0.E || desc->k != T0.k || desc->I != T0.I ||
      desc->S != T0.S || desc->dtype != T0.dtype)
    return MOE_ERR_INVALID_ARG;
  if (desc->T == 0) return MOE_OK;
  if (!x || !Wr || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(y) || (residual && !aligned16(residual)) ||
      (topk_ids_out && !aligned16(topk_ids_out)) || (topk_w_out && !aligned16(topk_w_out)))
    return MOE_ERR_INVALID_ARG;
  if (sel_bias && desc->gate != MOE_GATE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(desc, workspace, ws_bytes)) != MOE_OK) return st;
  std::lock_guard<std::mutex> g(tier->mu);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Ws W = carve(workspace, ws_layout(*desc));
  const int nE = tier->nE;
  const int P = desc->T * (desc->k + desc->S);
  int32_t* ids = topk_ids_out ? topk_ids_out : W.topk_ids;
  float* w = topk_w_out ? topk_w_out : W.topk_w;
  if (tier->done_recorded && cudaStreamWaitEvent(s, tier->done, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemsetAsync(W.flags, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
  if ((st = route_and_plan(desc, x, Wr, logit_bias, sel_bias, ids, w, W, s)) != MOE_OK) return st;
  if (permute_rows(desc, false, x, W.offsets, W.tok_idx, W.slot_row, W, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  // the routing decision reaches the host: batch bounds per expert
  int32_t* bounds = tier->host_tab;
  if (cudaMemcpyAsync(bounds, W.offsets, (size_t)(nE + 1) * 4, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  std::vector<int32_t> active;
  for (int e = 0; e < nE; ++e)
    if (bounds[e + 1] > bounds[e]) active.push_back(e);
  const int n = (int)active.size();
  std::vector<int32_t> slot(n), load(n), pass(n);
  int32_t n_passes = 0;
  if (!tier->cache.assign(active.data(), n, slot.data(), load.data(), pass.data(), &n_passes))
    return MOE_ERR_DEVICE_INPUT;  // batch bounds that are not a partition
  const double mean_rows = (double)P / (double)nE;
  for (int p = 0; p < n_passes; ++p) {
    int32_t* tab = tier->host_tab + (nE + 1) + (size_t)p * nE;
    for (int e = 0; e < nE; ++e) tab[e] = -1;
    for (int i = 0; i < n; ++i)
      if (pass[i] == p) tab[active[i]] = slot[i];
    int32_t* dtab = tier->dev_tab + (size_t)p * nE;
    if (cudaMemcpyAsync(dtab, tab, (size_t)nE * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if ((st = tier_load_all(tier, active.data(), slot.data(), load.data(), pass.data(), n, p,
                            s)) != MOE_OK)
      return st;
    if (launch_ffn_tc(W.x_perm, W.offsets, nE, P, desc->d, desc->I, mean_rows, tier->pool[0],
                      tier->pool[1], tier->pool[2], nullptr, W.h, W.y_perm, W.flags, s,
                      tier->n_slots, dtab) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (launch_combine(desc->dtype, W.y_perm, W.slot_row, w, residual, desc->T, desc->d, desc->k,
                     desc->S, y, s) != cudaSuccess ||
      cudaEventRecord(tier->done, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  tier->done_recorded = true;
  return MOE_OK;
}

moe_status moe_check_bounded_wait(void* workspace, size_t ws_bytes, int which, void* stream) {
  if (!workspace || ws_bytes < 16 || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  if (which < 0 || which > 3) return MOE_ERR_INVALID_ARG;
  return launch_bounded_wait_check(which, static_cast<int*>(workspace),
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_get_device_status(void* workspace, size_t ws_bytes, int clear, void* stream) {
  if (!workspace || ws_bytes < 16 || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host_flags[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(host_flags, workspace, sizeof(host_flags), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (clear && cudaMemsetAsync(workspace, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (host_flags[0] & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (host_flags[0] & kErrDeviceInput) return MOE_ERR_DEVICE_INPUT;
  return MOE_OK;
}

const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: bad pointer, size, alignment or flag";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape or dtype not supported";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded wait inside a kernel expired";
    case MOE_ERR_DEVICE_INPUT: return "MOE_ERR_DEVICE_INPUT: an input value was out of range";
  }
  return "unknown moe_status";
}

int64_t moe_launch_count(void) { return g_launches.load(); }

moe_status moe_profile_enable(int on) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (auto& r : g_prof) {
    g_prof_free.push_back(r.start);
    g_prof_free.push_back(r.stop);
  }
  g_prof.clear();
  g_prof_on = on != 0;
  g_prof_bytes_only = on == 2;
  return MOE_OK;
}

moe_status moe_profile_query(const char* kernel, int32_t* launches, float* total_ms) {
  if (!kernel || !launches || !total_ms) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_prof_mu);
  int n = 0;
  float tot = 0.f;
  for (auto& r : g_prof) {
    if (r.name != kernel) continue;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return MOE_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return MOE_ERR_CUDA;
    tot += ms;
    ++n;
  }
  *launches = n;
  *total_ms = tot;
  return MOE_OK;
}

moe_status moe_profile_list(const char* kernel, int32_t max_n, float* ms, uint64_t* bytes,
                            int32_t* n_out) {
  if (!kernel || !n_out || max_n < 0 || (max_n > 0 && (!ms || !bytes)))
    return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_prof_mu);
  int n = 0;
  for (auto& r : g_prof) {
    if (r.name != kernel) continue;
    if (n < max_n) {
      if (cudaEventSynchronize(r.stop) != cudaSuccess) return MOE_ERR_CUDA;
      float t = 0.f;
      if (cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) return MOE_ERR_CUDA;
      ms[n] = t;
      bytes[n] = r.bytes;
    }
    ++n;
  }
  *n_out = n;
  return MOE_OK;
}

}  // extern "C"
