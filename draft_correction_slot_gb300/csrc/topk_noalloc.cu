// topk_noalloc.cu -- step 1 (per-slot top-K) for callers that cannot
// allocate device memory.
//
// The handle-based entry points get their scratch from dcoco_create, which
// calls cudaMalloc.  Some callers cannot do that: a plugin running inside a
// serving engine that reserved all device memory for its own pool up front,
// or code on a latency-critical path where a cudaMalloc (which can
// synchronise the device) is not acceptable.  dcoco_topk_noalloc runs the
// same top-K kernel with its scratch -- per-row segment lists, finished-segment
// counters -- in the fixed array below, which every
// GPU that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/dcoco.h"
#include "kernels.h"

namespace {

constexpr int kMaxRows = DCOCO_TOPK_NOALLOC_MAX_ROWS;          // batch * (slots - 1)
constexpr size_t kScratchBytes = (size_t)4 << 20;              // 4 MiB
constexpr size_t kCountOff = 0;                                // unsigned [kMaxRows]
constexpr size_t kPartOff = (size_t)kMaxRows * 4;              // u64 segment lists
constexpr size_t kPartEntries = (kScratchBytes - kPartOff) / 8;
static_assert(kPartOff % 256 == 0, "aligned sub-arrays");

// The scratch.  In host code this name is only a stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_topk_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// Per device: the top-K occupancy (resident CTAs on the device for K = 8,
// 16, 32), then the device address of g_topk_scratch.  The address is
// published with release order after the occupancy is written, and read
// with acquire order, so a thread that sees the address also sees the
// occupancy.
int g_wave[kMaxDevices][3];
std::atomic<unsigned char *> g_scratch[kMaxDevices];

int k_index(int K) { return K == 8 ? 0 : (K == 16 ? 1 : 2); }

// Once per device, with that device current: look up the scratch address and
// the top-K occupancy.  Returns DCOCO_OK or DCOCO_ECUDA.
int setup_device(int dev) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch[dev].load(std::memory_order_acquire)) return DCOCO_OK;
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return DCOCO_ECUDA;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return DCOCO_ECUDA;
  }
  const int ks[3] = {8, 16, 32};
  for (int j = 0; j < 3; ++j) g_wave[dev][j] = sms * dc::topk_occupancy(ks[j]);
  g_scratch[dev].store(static_cast<unsigned char *>(p), std::memory_order_release);
  return DCOCO_OK;
}

// Argument checks that need no CUDA call.  The segment lists of a call take
// rows * topk * segments entries of the fixed list area; a call whose rows
// do not fit even at the fewest segments the vocabulary allows is rejected.
int check_args(int batch, int slots, int vocab, int topk) {
  if (slots < 3 || slots > 32 || (topk != 8 && topk != 16 && topk != 32)) return DCOCO_EUNSUPPORTED;
  if (vocab < topk || vocab > (1 << 20)) return DCOCO_EINVAL;
  if (batch < 0 || (long long)batch * (slots - 1) > kMaxRows) return DCOCO_EBATCH;
  if (batch == 0) return DCOCO_OK;
  const long long fit = (long long)kPartEntries / ((long long)batch * (slots - 1) * topk);
  if (fit < dc::topk_min_segments(vocab)) return DCOCO_EBATCH;
  return DCOCO_OK;
}

// The segment plan of a call on the current device: the plan the handle-based
// entry would take, limited to what the fixed list area holds.
int noalloc_plan(int batch, int slots, int vocab, int topk, dc::TopkPlan *plan, int *planned) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DCOCO_ECUDA;
  if (!g_scratch[dev].load(std::memory_order_acquire)) {
    const int rc = setup_device(dev);
    if (rc != DCOCO_OK) return rc;
  }
  const int rows = batch * (slots - 1);
  *plan = dc::topk_plan(vocab, rows, g_wave[dev][k_index(topk)]);
  *planned = plan->nchunks;
  const long long fit = (long long)kPartEntries / ((long long)rows * topk);
  if (plan->nchunks > fit) {
    plan->nchunks = (int)fit;
    const int nvec = vocab >> 3;
    plan->chunk_vecs = (nvec + plan->nchunks - 1) / plan->nchunks;
  }
  return DCOCO_OK;
}

}  // namespace

extern "C" int dcoco_topk_noalloc_plan(int batch, int slots, int vocab, int topk, int *segments,
                                       int *planned_segments) {
  if (!segments || !planned_segments) return DCOCO_EINVAL;
  int rc = check_args(batch, slots, vocab, topk);
  if (rc != DCOCO_OK) return rc;
  if (batch == 0) {
    *segments = *planned_segments = 0;
    return DCOCO_OK;
  }
  dc::TopkPlan plan;
  rc = noalloc_plan(batch, slots, vocab, topk, &plan, planned_segments);
  if (rc != DCOCO_OK) return rc;
  *segments = plan.nchunks;
  return DCOCO_OK;
}

extern "C" int dcoco_topk_noalloc(int batch, int slots, int vocab, int topk, const void *logits,
                                  int64_t logits_slot_stride, int32_t *topk_ids, float *topk_val,
                                  void *stream) {
  int rc = check_args(batch, slots, vocab, topk);
  if (rc != DCOCO_OK || batch == 0) return rc;
  if (!logits || !topk_ids || !topk_val) return DCOCO_EINVAL;
  if (logits_slot_stride < vocab || logits_slot_stride % 8 != 0 ||
      (reinterpret_cast<uintptr_t>(logits) & 15u) != 0)
    return DCOCO_EINVAL;
  dc::TopkPlan plan;
  int planned = 0;
  rc = noalloc_plan(batch, slots, vocab, topk, &plan, &planned);
  if (rc != DCOCO_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DCOCO_ECUDA;
  unsigned char *base = g_scratch[dev].load(std::memory_order_acquire);
  const int rows = batch * (slots - 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned *row_count = reinterpret_cast<unsigned *>(base + kCountOff);
  unsigned long long *part = reinterpret_cast<unsigned long long *>(base + kPartOff);
  // The array keeps the previous call's contents: the counters must start
  // at zero.
  if (cudaMemsetAsync(row_count, 0, (size_t)rows * sizeof(unsigned), st) != cudaSuccess)
    return DCOCO_ECUDA;
  // No programmatic overlap with the caller's previous kernel, which may
  // still be writing the logits.
  const cudaError_t e = dc::launch_topk(topk, static_cast<const uint16_t *>(logits), logits_slot_stride,
                                        slots, batch, vocab, plan, part, row_count, topk_ids, topk_val, st, false);
  return e == cudaSuccess ? DCOCO_OK : DCOCO_ECUDA;
}
