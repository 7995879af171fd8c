// noalloc.cu -- fia_decode_run_noalloc: the decode branch of fia_run for
// callers that cannot provide a workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code that executes while another component owns every byte of
// the device through its own pool, plugins whose host process forbids
// allocations after start-up, or real-time paths that must not take the
// allocator's locks or latency.  They still own q, the KV cache and the
// outputs, but have no way to obtain the scheduler's scratch (the work plan,
// the chunk claim queue and the partial (m, l, acc) slots).  This entry point
// uses a fixed scratch array compiled into the library instead: a file-scope
// __device__ array of FIA_NOALLOC_SCRATCH_BYTES, which every GPU that loads
// libfia holds from module load until the process exits.
//
// The array is shared by all calls on a device and keeps the previous call's
// contents.  Everything that must start at zero is cleared by the call itself
// (the scheduler kernel resets the error word and the claim counters), so
// a stale plan never leaks into a new call; but two calls whose work
// overlaps on the GPU (different streams without ordering) race on the array.
// The array's first int32 is the run's error word; the caller gets a copy of
// it through `status`, since it has no address of its own for the array.
#include "../../include/fia.h"
#include "internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[FIA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress.  It is looked up on every call: after a device reset
// or in another context on the same device the module is loaded again, at
// another address, and a cached pointer would dangle.
fia_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FIA_ERR_CUDA;
  *out = p;
  return FIA_OK;
}

}  // namespace

extern "C" fia_status fia_decode_run_noalloc(const fia_params* p, int32_t* status, void* stream) {
  fia::NvtxRange range("fia_decode_run_noalloc");
  fia_plan_layout lay;
  fia_status st = fia_get_plan_layout(p, &lay);
  if (st != FIA_OK) return st;
  if (lay.branch == 2) return FIA_ERR_UNSUPPORTED;  // decode only
  if (lay.total_bytes > (int64_t)FIA_NOALLOC_SCRATCH_BYTES) return FIA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (lay.branch == 0) {  // no query row: nothing runs, and nothing failed
    if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess)
      return FIA_ERR_CUDA;
    return FIA_OK;
  }
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != FIA_OK) return st;
  st = fia_run(p, scratch, FIA_NOALLOC_SCRATCH_BYTES, stream);
  if (st != FIA_OK) return st;
  if (status && cudaMemcpyAsync(status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
                    cudaSuccess)
    return FIA_ERR_CUDA;
  return FIA_OK;
}
