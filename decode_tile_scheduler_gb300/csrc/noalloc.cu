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
#include <mutex>

#include "../../include/fia.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[FIA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address has to come from
// cudaGetSymbolAddress, looked up once per device with that device current.
fia_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FIA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FIA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FIA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return FIA_OK;
}

}  // namespace

extern "C" fia_status fia_decode_run_noalloc(const fia_params* p, void* stream) {
  fia_plan_layout lay;
  fia_status st = fia_get_plan_layout(p, &lay);
  if (st != FIA_OK) return st;
  if (lay.branch != 1 && lay.total_bytes > 256) return FIA_ERR_UNSUPPORTED;  // decode only
  if (lay.total_bytes > (int64_t)FIA_NOALLOC_SCRATCH_BYTES) return FIA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != FIA_OK) return st;
  return fia_run(p, scratch, FIA_NOALLOC_SCRATCH_BYTES, stream);
}
