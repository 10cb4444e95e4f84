// Token selection (lm_head + greedy argmax) that allocates nothing and needs
// no bound workspace.
//
// Some callers cannot hand this library device memory: a host that embeds the
// draft head in a process whose device memory is owned by another runtime (a
// serving engine's caching allocator or a graph-capture pool it cannot
// extend), or a plugin that may not call cudaMalloc at all.  For them this
// entry point keeps its scratch -- the argmax keys of the rows, the stream-K
// partial tiles and per-tile tickets of the tensor-core GEMM, and a device
// status word -- in one file-scope __device__ array that every GPU which
// loads the library holds until the process exits.
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/dflash.h"
#include "common.cuh"
#include "kernels.h"

using namespace dflash;

namespace {

constexpr int kNoAllocMaxRows = 32;                    // rows per call (token tile <= 32)
constexpr int kNoAllocMaxTiles = 2048;                 // 128-row vocabulary tiles (vocab <= 262144)
constexpr size_t kErrOff = 0;
constexpr size_t kKeysOff = 256;
constexpr size_t kTicketsOff = kKeysOff + 8 * kNoAllocMaxRows;
constexpr size_t kPartialsOff = kTicketsOff + 4 * (size_t)kNoAllocMaxTiles;
// stream-K partials: per persistent CTA two slots of (token tile x 128) fp32
constexpr size_t kPartialsBytes = (size_t)kTcMaxCtas * 2 * kNoAllocMaxRows * 128 * 4;
constexpr size_t kScratchBytes = kPartialsOff + kPartialsBytes;   // about 5.3 MB

}  // namespace

// The scratch itself.  Host code must not use this symbol as an address: it
// is a host-side stand-in.  The device address comes from
// cudaGetSymbolAddress at set-up.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char *g_scratch_ptr[kMaxDevices] = {};

// keys -> token ids.  A call whose bounded waits gave up (its status word is
// non-zero) reports -1 ids rather than ids built from unmerged partial tiles,
// and copies the word to the caller's status.
__global__ void keys_to_ids_kernel(const unsigned long long *__restrict__ keys, int rows,
                                   const unsigned int *__restrict__ err, int *__restrict__ ids,
                                   unsigned int *__restrict__ status) {
  pdl_wait();
  const unsigned int word = __ldcg(err);
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < rows) ids[r] = word ? -1 : argmax_key_index(keys[r]);
  if (status && r == 0) *status = word;
}

int noalloc_fail(int st, const char *msg) {
  set_last_error(msg);
  return st;
}

// Once per device, with that device current: the device address of the
// scratch and the tensor-core kernels' shared-memory limits.
int setup_device(unsigned char **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return noalloc_fail(DFLASH_ECUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(DFLASH_EUNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return noalloc_fail(DFLASH_ECUDA, "cudaGetSymbolAddress of the no-alloc scratch failed");
    if (prepare_gemm_tc() != cudaSuccess)
      return noalloc_fail(DFLASH_ECUDA, "setting tensor-core GEMM attributes failed");
    g_scratch_ptr[dev] = (unsigned char *)ptr;
  }
  *out = g_scratch_ptr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_select_tokens_noalloc(dflash_handle *h, int32_t rows, const void *hidden,
                                            int32_t *ids, uint32_t *status,
                                            dflash_stream_t stream) {
  if (!h || !hidden || !ids) return noalloc_fail(DFLASH_EINVAL, "handle, hidden and ids must be non-NULL");
  const void *lm_head = nullptr;
  int H = 0, V = 0, dtype = 0;
  if (handle_lm_head(h, &lm_head, &H, &V, &dtype) != DFLASH_OK)
    return noalloc_fail(DFLASH_EINVAL, "invalid handle");
  if (dtype != DFLASH_BF16) return noalloc_fail(DFLASH_EUNSUPPORTED, "bf16 configurations only");
  if (rows < 0) return noalloc_fail(DFLASH_EINVAL, "negative rows");
  if (rows == 0) return DFLASH_OK;
  if (rows > kNoAllocMaxRows) return noalloc_fail(DFLASH_ECAPACITY, "rows > 32");
  const int tiles = (V + 127) / 128;
  if (tiles > kNoAllocMaxTiles) return noalloc_fail(DFLASH_ECAPACITY, "vocab > 262144");
  // the GEMM reads hidden through a tensor map (16-byte aligned rows) in
  // k-blocks of 64 features
  if ((uintptr_t)hidden % 16 != 0) return noalloc_fail(DFLASH_EINVAL, "hidden must be 16-byte aligned");
  if (H % 64 != 0) return noalloc_fail(DFLASH_EUNSUPPORTED, "hidden size must be a multiple of 64");
  cudaStream_t s = (cudaStream_t)stream;
  unsigned char *scratch = nullptr;
  if (int st = setup_device(&scratch)) return st;
  unsigned long long *keys = (unsigned long long *)(scratch + kKeysOff);
  unsigned int *err = (unsigned int *)(scratch + kErrOff);
  // The array keeps the previous call's contents: the status word, the argmax
  // keys and the per-tile tickets (a call whose waits gave up can leave a
  // ticket non-zero) all start from zero.  They are contiguous.
  static_assert(kErrOff == 0 && kKeysOff < kTicketsOff, "cleared region layout");
  if (cudaMemsetAsync(scratch, 0, kTicketsOff + 4 * (size_t)tiles, s) != cudaSuccess)
    return noalloc_fail(DFLASH_ECUDA, "clearing the no-alloc scratch failed");
  GemmProblem P;
  std::memset(&P, 0, sizeof(P));
  P.A.ptr[0] = hidden;
  P.A.ld = H;
  P.A.k_per_src = H;
  P.A.n_src = 1;
  P.M = rows;
  P.K = H;
  GemmSeg &g = P.seg[P.nseg++];
  g.W = lm_head;
  g.ldw = H;
  g.N = V;
  std::memset(&g.epi, 0, sizeof(g.epi));
  g.epi.op = EPI_ARGMAX;
  g.epi.N = V;
  g.epi.argmax_keys = keys;
  if (launch_gemm_tc(P, (float *)(scratch + kPartialsOff), (int *)(scratch + kTicketsOff),
                     kNoAllocMaxTiles, err, s) != cudaSuccess)
    return noalloc_fail(DFLASH_ECUDA, "lm_head GEMM launch failed");
  if (launch_pdl(keys_to_ids_kernel, dim3((rows + 127) / 128), dim3(128), 0, s,
                 (const unsigned long long *)keys, (int)rows, (const unsigned int *)err, (int *)ids,
                 (unsigned int *)status) != cudaSuccess)
    return noalloc_fail(DFLASH_ECUDA, "argmax id kernel launch failed");
  return DFLASH_OK;
}
