// eagle_lm_head_topk_noalloc: the fused LM-head top-k for callers that cannot allocate
// device memory.
//
// Who needs it: a serving engine that reserves nearly all of HBM for its own KV-cache
// pool at start-up and forbids any later cudaMalloc; a latency-critical decode loop in
// which cudaMalloc / cudaFree would synchronise the device and stall the other streams;
// a program with a fixed device-memory budget decided before it loads this library.
// Such callers cannot create an eagle_draft_t handle (its workspace is cudaMalloc'd), so
// this entry point takes the weights, inputs and outputs as plain device pointers and
// keeps the kernels' scratch in one file-scope __device__ array instead.
//
// The scratch array (4 MiB) is held on every GPU that loads the library until the process
// exits.  All calls share it and it keeps the last call's contents: a call clears what
// must start at zero (the split-K arrival counters and the error word), and two calls
// whose kernels overlap on the GPU (different streams or host threads) race on it.
//
// Errors inside the kernels: there is no handle to carry a device error word to the host,
// so the call reports through its outputs.  If a bounded wait in the LM-head kernel runs
// out, the tiles it never reached would leave the previous call's partials in the array;
// the merge kernel then writes id -1 and NaN log-probability / log-sum-exp for every row
// rather than merging them.  A row whose logits are not finite gets id -1 for each of the
// k places it could not fill.
#include "../../include/eagle_draft.h"
#include "common.cuh"
#include "internal.h"

#include <cstdio>
#include <cstring>
#include <mutex>

using namespace eagle;

namespace {

constexpr int NA_MAX_ROWS = 16;
constexpr int NA_MAX_K = 16;
constexpr int NA_MAX_VOCAB = 131072;
constexpr int NA_MAX_D = 16384;
constexpr int NA_MAX_CTAS = 192;
constexpr int NA_MAX_TILES = NA_MAX_VOCAB / BM;
constexpr size_t NA_SCRATCH_BYTES = size_t(4) << 20;

// byte offsets inside the scratch array
constexpr size_t NA_PART = 0;                                                     // split-K partial tiles
constexpr size_t NA_PART_BYTES = size_t(NA_MAX_CTAS) * 2 * NA_MAX_ROWS * BM * 4;
constexpr size_t NA_COUNTERS = NA_PART + NA_PART_BYTES;                           // per-tile arrival counters
constexpr size_t NA_ERR = NA_COUNTERS + size_t(NA_MAX_TILES) * 4;                 // device error word
constexpr size_t NA_ZERO_BYTES = NA_ERR + 256 - NA_COUNTERS;                      // cleared by every call
constexpr size_t NA_LMMAX = NA_COUNTERS + NA_ZERO_BYTES;                          // per tile: max logit
constexpr size_t NA_LMSUM = NA_LMMAX + size_t(NA_MAX_TILES) * NA_MAX_ROWS * 4;    // per tile: sum of exp
constexpr size_t NA_LMVAL = NA_LMSUM + size_t(NA_MAX_TILES) * NA_MAX_ROWS * 4;    // per CTA: top-k values
constexpr size_t NA_LMID = NA_LMVAL + size_t(NA_MAX_CTAS) * NA_MAX_ROWS * NA_MAX_K * 4;
constexpr size_t NA_END = NA_LMID + size_t(NA_MAX_CTAS) * NA_MAX_ROWS * NA_MAX_K * 4;
static_assert(NA_END <= NA_SCRATCH_BYTES, "scratch layout exceeds the array");

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_SCRATCH_BYTES];

static std::mutex g_setup_mu;
static void* g_scratch_addr[256];   // per device ordinal: device address of g_noalloc_scratch

static eagle_status_t na_fail(eagle_status_t st, const char* msg) {
  set_last_error(msg);
  return st;
}

// Set-up, once per device and with that device current: the device address of the
// scratch array (its name in host code is only a host-side stand-in) and the kernels'
// shared-memory limits.
static eagle_status_t na_setup(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_addr[dev]) {
    *out = g_scratch_addr[dev];
    return EAGLE_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
    return na_fail(EAGLE_ERR_CUDA, "noalloc: cudaGetSymbolAddress of the scratch array failed");
  if (gemm_setup_attributes() != cudaSuccess || tree_setup_attributes() != cudaSuccess)
    return na_fail(EAGLE_ERR_CUDA, "noalloc: cudaFuncSetAttribute failed");
  g_scratch_addr[dev] = p;
  *out = p;
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_lm_head_topk_noalloc(const void* w_lm, int32_t vocab, int32_t d, const float* a,
                                                     int32_t N, int32_t k, int32_t* ids, float* logp, float* lse,
                                                     void* stream) {
  if (!w_lm || !a || !ids || !logp || !lse) return na_fail(EAGLE_ERR_INVALID_ARG, "noalloc: null pointer argument");
  if (N < 1 || N > NA_MAX_ROWS) return na_fail(EAGLE_ERR_INVALID_ARG, "noalloc: N must be 1..16 rows");
  if (k < 1 || k > NA_MAX_K) return na_fail(EAGLE_ERR_INVALID_ARG, "noalloc: k must be 1..16");
  if (vocab < BM || vocab > NA_MAX_VOCAB || vocab % BM)
    return na_fail(EAGLE_ERR_INVALID_ARG, "noalloc: vocab must be a multiple of 128 and at most 131072");
  if (d < BM || d > NA_MAX_D || d % BM)
    return na_fail(EAGLE_ERR_INVALID_ARG, "noalloc: d must be a multiple of 128 and at most 16384");
  if (reinterpret_cast<uintptr_t>(w_lm) % 16 || reinterpret_cast<uintptr_t>(a) % 16)
    return na_fail(EAGLE_ERR_INVALID_ARG, "noalloc: w_lm and a must be 16-byte aligned");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return na_fail(EAGLE_ERR_CUDA, "noalloc: cudaGetDevice");
  if (num_sms() > NA_MAX_CTAS) return na_fail(EAGLE_ERR_UNSUPPORTED, "noalloc: more than 192 SMs");
  void* base = nullptr;
  eagle_status_t st = na_setup(dev, &base);
  if (st != EAGLE_OK) return st;
  unsigned char* s = static_cast<unsigned char*>(base);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  GemmPlan p;
  p.tc = true;
  if (!make_weight_map(&p.tm0, w_lm, vocab, d)) return na_fail(EAGLE_ERR_CUDA, "noalloc: cuTensorMapEncodeTiled failed");
  p.tm1 = p.tm0;
  GemmArgs& g = p.args;
  memset(&g, 0, sizeof(g));
  g.M = vocab;
  g.K = d;
  g.m_split = vocab;
  g.part = reinterpret_cast<float*>(s + NA_PART);
  g.counters = reinterpret_cast<int*>(s + NA_COUNTERS);
  g.err = reinterpret_cast<unsigned*>(s + NA_ERR);
  g.b.mode = B_F32;
  g.b.x = a;
  g.b.ldx = d;
  g.e.kind = EPI_LMHEAD;
  g.e.lm_max = reinterpret_cast<float*>(s + NA_LMMAX);
  g.e.lm_sum = reinterpret_cast<float*>(s + NA_LMSUM);
  g.e.lm_val = reinterpret_cast<float*>(s + NA_LMVAL);
  g.e.lm_id = reinterpret_cast<int*>(s + NA_LMID);
  g.e.topk = k;
  if (!plan_gemm(p, N)) return na_fail(EAGLE_ERR_UNSUPPORTED, "noalloc: LM-head launch does not fit");
  if (p.grid > NA_MAX_CTAS || g.nrb * g.npad > NA_MAX_ROWS)
    return na_fail(EAGLE_ERR_UNSUPPORTED, "noalloc: launch needs more scratch than the array holds");

  if (cudaMemsetAsync(s + NA_COUNTERS, 0, NA_ZERO_BYTES, cs) != cudaSuccess)
    return na_fail(EAGLE_ERR_CUDA, "noalloc: clearing the counters failed");
  if (launch_gemm(p, cs, false) != cudaSuccess) return na_fail(EAGLE_ERR_CUDA, "noalloc: LM-head kernel launch failed");
  LmPartials lm;
  lm.max = g.e.lm_max;
  lm.sum = g.e.lm_sum;
  lm.val = g.e.lm_val;
  lm.id = g.e.lm_id;
  lm.G = p.grid;
  lm.T = vocab / BM;
  lm.poison_if = g.err;   // a wait that ran out leaves stale partials: poison the outputs instead
  if (launch_lm_merge(lm, N, k, ids, logp, lse, cs, false) != cudaSuccess)
    return na_fail(EAGLE_ERR_CUDA, "noalloc: merge kernel launch failed");
  return EAGLE_OK;
}
