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
// The host needs the array's device address to pass it to the kernels; the
// first call on each device looks it up with cudaGetSymbolAddress (with that
// device current) and caches it.  Make that first call before any stream
// capture.  No call allocates memory.
#include <cmath>
#include <cstring>

#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

constexpr int kNoAllocMaxVocab = 262144;
constexpr int kNoAllocStats = kMaxRows * ((kNoAllocMaxVocab + kVChunk - 1) / kVChunk);

static __device__ __align__(256) RowStat g_residual_stats[kNoAllocStats];
static_assert(sizeof(g_residual_stats) == 272 * 1024, "the size the header documents");

namespace {

constexpr int kMaxDevices = 64;
RowStat* g_stats_addr[kMaxDevices] = {nullptr};

// Device address of g_residual_stats on the current device (looked up once).
int stats_address(RowStat** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TV_E_CUDA;
  if (!g_stats_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_residual_stats) != cudaSuccess || !p) return TV_E_CUDA;
    g_stats_addr[dev] = static_cast<RowStat*>(p);
  }
  *out = g_stats_addr[dev];
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
  if (!trees || n_req < 1 || n_req > kMaxReq) return n_req < 1 || n_req > kMaxReq ? TV_E_ROWS : TV_E_ARG;
  ReqTable t;
  memset(&t, 0, sizeof(t));
  t.n_req = n_req;
  int total = 0;
  for (int r = 0; r < n_req; ++r) {
    const int n = trees[r].n;
    if (n < 1 || n > kMaxRows) return TV_E_ROWS;
    if (!trees[r].parent || !trees[r].token) return TV_E_ARG;
    t.row_off[r] = total;
    t.n[r] = n;
    t.parent[r] = trees[r].parent;
    t.token[r] = trees[r].token;
    total += n;
    if (total > kMaxRows) return TV_E_ROWS;
  }
  t.row_off[n_req] = total;
  t.total_rows = total;
  RowStat* stats = nullptr;
  const int rc = stats_address(&stats);
  if (rc != TV_OK) return rc;
  return launch_accept_residual(t, logits, vocab, temperature, uniforms, bonus_at_leaf ? 1 : 0, stats, path,
                                accept_len, out_tokens, out_count, dev_status, reinterpret_cast<cudaStream_t>(stream));
}
