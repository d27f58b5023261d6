// tv_accept_residual_noalloc: the residual-sampling accept walk for callers
// that cannot hand the library a workspace.
//
// tv_accept_residual keeps its per-row softmax statistics in caller-provided
// workspace memory.  Some callers have no way to get that memory: code that
// runs as a plugin step inside another framework's executor, where the host
// framework owns every device allocation and forbids cudaMalloc in the step;
// real-time loops with a no-allocation rule (cudaMalloc can synchronise the
// device and stall other streams); and callers that only hold a stream and the
// round's input/output buffers.  This entry point runs the same two kernels
// with the statistics in a fixed-size array that lives in the library's own
// device image instead.
//
// The array is a file-scope __device__ global: every GPU that loads the
// library holds one copy (272 KB) until the process exits.  Its size fixes the
// largest vocabulary this entry point accepts (kNoAllocMaxVocab); larger
// vocabularies are rejected with TV_E_UNSUPPORTED.  Nothing in it needs to
// start at zero: every statistic the walk reads is written earlier in the same
// call.  It keeps the previous call's contents until then, and all calls on a
// device share it, so two calls whose kernels overlap on the GPU (different
// streams without ordering between them) race on it.
//
// The host needs the array's device address to pass it to the kernels.  Each
// call looks it up with cudaGetSymbolAddress in the context current on the
// calling thread: a host-side table lookup that allocates nothing.  Nothing is
// cached, so a call made after cudaDeviceReset, or with another context
// current (a host framework's own driver-API context), gets that context's
// copy of the array and never a stale address.  The first call in a context
// also loads the library's device image there: make that call before any
// stream capture.  No call allocates memory.
#include <cmath>

#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

constexpr int kNoAllocMaxVocab = 262144;
constexpr int kNoAllocStats = kMaxRows * ((kNoAllocMaxVocab + kVChunk - 1) / kVChunk);

static __device__ __align__(256) RowStat g_residual_stats[kNoAllocStats];
static_assert(sizeof(g_residual_stats) == 272 * 1024, "the size the header documents");

namespace {

// Device address of g_residual_stats in the current context.
int stats_address(RowStat** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_residual_stats) != cudaSuccess || !p) return TV_E_CUDA;
  *out = static_cast<RowStat*>(p);
  return TV_OK;
}

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" int tv_accept_residual_noalloc(const tv_tree* trees, int n_req, const float* logits, int32_t vocab,
                                          float temperature, const float* uniforms, int bonus_at_leaf,
                                          int32_t* path, int32_t* accept_len, int32_t* out_tokens,
                                          int32_t* out_count, int32_t* dev_status, void* stream) {
  if (!(std::isfinite(temperature) && temperature > 0.f)) return TV_E_TEMP;
  if (!logits || !uniforms || !path || !accept_len || !out_tokens || !out_count || !dev_status || vocab < 2)
    return TV_E_ARG;
  if (vocab > kNoAllocMaxVocab) return TV_E_UNSUPPORTED;
  ReqTable t;
  int rc = build_table(t, trees, nullptr, n_req, true);
  if (rc != TV_OK) return rc;
  RowStat* stats = nullptr;
  if ((rc = stats_address(&stats)) != TV_OK) return rc;
  return launch_accept_residual(t, logits, vocab, temperature, uniforms, bonus_at_leaf ? 1 : 0, stats, path,
                                accept_len, out_tokens, out_count, dev_status, reinterpret_cast<cudaStream_t>(stream));
}
