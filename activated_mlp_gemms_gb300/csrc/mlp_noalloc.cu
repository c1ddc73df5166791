// mlp_noalloc.cu -- mlp_fwd_infer_noalloc: the inference forward with its
// scratch in a fixed device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot hand the library a workspace because they
// may not allocate device memory when they run the MLP -- for example a C
// runtime whose device memory is planned once at start-up and frozen, or a
// serving loop that must not call cudaMalloc (it synchronises the device and
// stalls every other stream) and has no caching allocator to draw from.
//
// The scratch is the file-scope array below, MLP_NOALLOC_SCRATCH_BYTES long.
// It lives in every device that loads this library, from module load until
// the process exits.  Host code cannot use the array's name as a device
// address (in host code it names a host-side shadow), so every call fetches
// the array's device address on the current device with
// cudaGetSymbolAddress (cheap once the module is loaded; a cached address
// would go stale after a device reset).  Its first 4 bytes are the status
// word that mlp_noalloc_status reads.
#include "mlp.h"

namespace {

constexpr size_t kScratchBytes = MLP_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_for_current_device() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
  return ptr;
}

}  // namespace

extern "C" int mlp_fwd_infer_noalloc(const mlp_problem_t* p, const void* x, const void* Wg,
                                     const void* Wu, const void* Wd, void* out, void* stream) {
  const size_t need = mlp_workspace_size(p, MLP_MODE_INFER);
  if (need == 0) return MLP_ERR_INVALID_ARG;
  if (need > kScratchBytes) return MLP_ERR_WORKSPACE_TOO_SMALL;
  void* ws = scratch_for_current_device();
  if (!ws) return MLP_ERR_CUDA;
  // mlp_fwd_infer clears the status word and scheduler counters at the start
  // of the scratch on the stream, and overwrites the postact before reading it.
  return mlp_fwd_infer(p, x, Wg, Wu, Wd, out, ws, kScratchBytes, stream);
}

extern "C" int mlp_noalloc_status(void* stream) {
  void* ws = scratch_for_current_device();
  if (!ws) return MLP_ERR_CUDA;
  return mlp_device_status(ws, stream);
}
