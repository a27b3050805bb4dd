// Host-side state that the launchers look up on every call, cached per CUDA
// context so that a launch costs one small table lookup instead of a round of
// runtime queries.
//
// The key is the driver's context id (cuCtxGetId), which is unique for the
// life of the process: a device reset or a context created later gets a new
// id, so nothing cached for an old context is ever used in a new one.  When
// no context is current yet (no runtime call has run on this thread) or the
// id cannot be read, the caller's query runs uncached.
#include <cuda.h>

#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {
namespace {

using CtxGetCurrent = CUresult (*)(CUcontext *);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long *);

struct DriverFns {
  CtxGetCurrent get_current = nullptr;
  CtxGetId get_id = nullptr;
};

const DriverFns &driver_fns() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetId>(f);
  });
  return fns;
}

// One cached fact about a kernel (or the device) in one context.
struct Entry {
  uint64_t ctx;
  const void *kern;  // null for per-device facts
  int kind;          // what `value` is
  int arg;           // shared memory bytes of an occupancy query, else 0
  int value;
};
enum { kSmemSet = 0, kSmCount = 1, kOccupancy = 2 };

std::mutex g_mu;
std::vector<Entry> g_entries;
constexpr size_t kMaxEntries = 4096;  // old contexts' entries are dropped past this

bool lookup(uint64_t ctx, const void *kern, int kind, int arg, int *value) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (const Entry &e : g_entries)
    if (e.ctx == ctx && e.kern == kern && e.kind == kind && e.arg == arg) {
      *value = e.value;
      return true;
    }
  return false;
}

// Sets (or adds) the entry's value.
void remember(uint64_t ctx, const void *kern, int kind, int arg, int value) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (Entry &e : g_entries)
    if (e.ctx == ctx && e.kern == kern && e.kind == kind && e.arg == arg) {
      e.value = value;
      return;
    }
  if (g_entries.size() >= kMaxEntries) g_entries.clear();
  g_entries.push_back(Entry{ctx, kern, kind, arg, value});
}

}  // namespace

uint64_t current_context_id() {
  const DriverFns &fns = driver_fns();
  if (fns.get_current == nullptr || fns.get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id == 0 ? 0 : static_cast<uint64_t>(id);
}

// A kernel has one shared-memory limit per context.  The cache keeps the
// value last set; a request at or under it needs no call, and a larger one
// raises the limit (a limit above a launch's size is harmless).  Check and
// set happen under one lock, so the limit only grows and no caller can lower
// it under another's launch.
cudaError_t set_max_smem(const void *kern, int smem) {
  static std::mutex mu;
  const uint64_t ctx = current_context_id();
  if (ctx == 0)
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  std::lock_guard<std::mutex> lock(mu);
  int limit = 0;
  if (lookup(ctx, kern, kSmemSet, 0, &limit) && smem <= limit) return cudaSuccess;
  const cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err == cudaSuccess) remember(ctx, kern, kSmemSet, 0, smem);
  return err;
}

cudaError_t sm_count(int *sms) {
  const uint64_t ctx = current_context_id();
  if (ctx != 0 && lookup(ctx, nullptr, kSmCount, 0, sms)) return cudaSuccess;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (err == cudaSuccess && ctx != 0) remember(ctx, nullptr, kSmCount, 0, *sms);
  return err;
}

cudaError_t blocks_per_sm(int *n, const void *kern, int threads, int smem) {
  const uint64_t ctx = current_context_id();
  // threads is fixed per kernel here, so (kernel, smem) identifies the query
  if (ctx != 0 && lookup(ctx, kern, kOccupancy, smem, n)) return cudaSuccess;
  cudaError_t err = set_max_smem(kern, smem);
  if (err == cudaSuccess)
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, threads, smem);
  if (err == cudaSuccess && ctx != 0) remember(ctx, kern, kOccupancy, smem, *n);
  return err;
}

}  // namespace pa
