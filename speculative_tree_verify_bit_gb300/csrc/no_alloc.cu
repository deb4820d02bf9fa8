// no_alloc.cu -- verify attention plus split merge for callers that cannot
// allocate device memory.
//
// stv_verify_attn needs a caller-owned workspace for its per-split partial
// results.  Some callers cannot provide one: a serving engine that has
// already handed nearly all device memory to its own KV-page allocator (an
// extra cudaMalloc in the middle of a decode step can fail, or force the
// engine to shrink its cache), or a plain C host that has no device
// allocator of its own.  For them this file keeps the scratch in a
// library-owned, file-scope __device__ array of fixed size, so that the call
// needs only its inputs and its output.
//
// Cost and limits: every GPU on which this library's code is loaded holds
// kNoAllocScratchBytes of device memory for the array until the process
// exits.  All calls share the one array, so calls that overlap on the GPU
// (other streams, other host threads) race on it; serialise them.  The array
// keeps the previous call's contents; nothing in it has to start at zero,
// because the verify pass writes every partial before the merge reads it.
#include <mutex>

#include "stv_internal.h"

namespace stv {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_no_alloc_scratch[kNoAllocScratchBytes];

// Host code cannot use g_no_alloc_scratch's name as a device address (on the
// host it names a stand-in object).  The device address is looked up once
// per device, with that device current, and cached.
static std::mutex g_scratch_mutex;
static void* g_scratch_ptr[kMaxDevices] = {};

static int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return STV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || !p) return STV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return STV_OK;
}

}  // namespace stv

extern "C" int stv_verify_attn_no_alloc(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs,
                                        int n_seqs, const void* q, const int32_t* parent, int t_nodes, int path,
                                        void* o, int32_t* dev_status, stv_stream_t stream) {
  using namespace stv;
  if (!o) return STV_ERR_INVALID_ARG;
  size_t need = 0;
  int rc = stv_verify_workspace_bytes(shape, seqs, n_seqs, t_nodes, 0, &need);
  if (rc) return rc;
  if (need > kNoAllocScratchBytes) return STV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch))) return rc;
  rc = stv_verify_attn(shape, layer, seqs, n_seqs, q, parent, t_nodes, path, scratch, kNoAllocScratchBytes,
                       dev_status, stream);
  if (rc) return rc;
  return stv_split_combine(shape, seqs, n_seqs, t_nodes, scratch, kNoAllocScratchBytes, o, stream);
}
