// Tree acceptance with library-owned scratch (ds_accept_static).
//
// ds_accept needs a small device workspace: a status word for the sticky
// input-error bits and one NodeStats record per tree node, which the node
// pass writes and the walk reads.  Some callers cannot hand out device
// memory at the call site (a plugin or host callback whose framework owns
// every allocation and offers no allocator, or a serving loop that forbids
// allocation once it is warm).  For them this entry keeps that scratch in a
// fixed-size array in device global memory that belongs to this file, and
// runs the same two kernels as ds_accept over it.
//
// Nothing here allocates: the array is part of the loaded module, its
// address is looked up on every call (the lookup allocates nothing), and
// each call only enqueues a 256-byte memset of the status word and the
// acceptance kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ds.h"
#include "internal.h"

namespace ds {
namespace {

constexpr int kStaticNodes = DS_ACCEPT_STATIC_MAX_NODES;
constexpr size_t kStaticBytes = kStatusBytes + (size_t)kStaticNodes * sizeof(NodeStats);
static_assert(kStaticBytes % kAlign == 0, "scratch must be a whole number of 256-byte units");

// status word at byte 0, NodeStats records from byte kStatusBytes on: the
// same layout accept_layout() gives a caller's workspace
static __device__ __align__(256) unsigned char g_accept_scratch[kStaticBytes];

// Address of g_accept_scratch in the current context, looked up on every
// call: the lookup allocates nothing, and a context that was torn down and
// created again (cudaDeviceReset) never leaves a stale address behind.
ds_status scratch_for_current_device(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_accept_scratch);
  if (e != cudaSuccess || !p)
    return set_last_error(DS_ERR_CUDA,
                          "ds_accept_static: cudaGetSymbolAddress of the scratch failed");
  *out = p;
  return DS_OK;
}

}  // namespace
}  // namespace ds

extern "C" ds_status ds_accept_static(const ds_accept_args* args, uint32_t* flags_out,
                                      void* stream) {
  using namespace ds;
  if (!args) return set_last_error(DS_ERR_INVALID_ARG, "args is NULL");
  if (args->workspace || args->workspace_bytes)
    return set_last_error(DS_ERR_INVALID_ARG,
                          "ds_accept_static uses its own scratch: workspace must be NULL and "
                          "workspace_bytes 0 (use ds_accept to pass a workspace)");
  if (args->n_nodes > kStaticNodes)
    return set_last_error(DS_ERR_UNSUPPORTED,
                          "n_nodes exceeds DS_ACCEPT_STATIC_MAX_NODES (4096), the capacity "
                          "of ds_accept_static's scratch: use ds_accept with a workspace");
  void* scratch = nullptr;
  ds_status st = scratch_for_current_device(&scratch);
  if (st != DS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status bits are sticky (the kernels only OR into them): start each
  // call from zero so that *flags_out describes this call alone
  cudaError_t e = cudaMemsetAsync(scratch, 0, kStatusBytes, s);
  if (e != cudaSuccess)
    return set_last_error(DS_ERR_CUDA, "ds_accept_static: clearing the status word failed");
  ds_accept_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kStaticBytes;
  st = ds_accept(&a, stream);   // validates every other argument, then launches
  if (st != DS_OK || !flags_out) return st;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess)
    return set_last_error(DS_ERR_CUDA, "ds_accept_static: stream synchronize failed");
  e = cudaMemcpy(flags_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess)
    return set_last_error(DS_ERR_CUDA, "ds_accept_static: reading the status word failed");
  return DS_OK;
}
