// muon_normalize_noalloc: the Frobenius normalisation out = in / (||in||_F + eps)
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running under a memory pool or
// allocator that owns all device memory, plugins whose host framework forbids
// allocation inside its callbacks, and real-time loops that must not hit the
// allocator's synchronisation. The other entry points keep their scratch in a
// per-handle workspace that they allocate on first use; this one keeps it in
// the file-scope array below instead, so it allocates nothing at any call.
//
// Scratch: per-block partial sums of squares, per-matrix arrival tickets and
// per-matrix inverse norms, in g_noalloc_scratch. The array is part of the
// library's device image: every GPU that loads the library holds it
// (kNoAllocScratchBytes) until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/muon.h"
#include "elementwise.cuh"

using namespace muon;

namespace {

constexpr int kNoAllocMaxMatrices = MUON_NOALLOC_MAX_MATRICES;
constexpr int64_t kNoAllocMaxChunks = MUON_NOALLOC_MAX_ELEMENTS / kFlatChunk;  // partial sums
constexpr size_t kPartialBytes = static_cast<size_t>(kNoAllocMaxChunks) * sizeof(float);
constexpr size_t kTicketBytes = kNoAllocMaxMatrices * sizeof(int);
constexpr size_t kInvBytes = kNoAllocMaxMatrices * sizeof(float);
constexpr size_t kNoAllocScratchBytes = kPartialBytes + kTicketBytes + kInvBytes;
static_assert(kNoAllocMaxMatrices <= kEwMax, "one launch serves every matrix");
static_assert(MUON_NOALLOC_MAX_ELEMENTS % kFlatChunk == 0, "whole chunks");

// Partial sums first, then the tickets (which must be zero when a call starts), then the inverse norms.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// The scratch address per device, with the context it was looked up in: a context created again
// (after cudaDeviceReset, say) can load the module at another address, so a changed context
// triggers a fresh lookup.
struct ScratchSlot {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
ScratchSlot g_scratch_slot[kMaxDevices];
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get_current = nullptr;

void put(char* msg, int len, const char* text) {
  if (msg && len > 0) {
    strncpy(msg, text, static_cast<size_t>(len) - 1);
    msg[len - 1] = '\0';
  }
}

// Device address of g_noalloc_scratch on the current device, looked up once per device and
// context (the first call on a device does it). In host code the array's name is only a stand-in;
// kernels must get this address.
muon_status scratch_for_current_device(void** out, char* msg, int len) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    put(msg, len, "no current CUDA device");
    return MUON_ERR_CUDA;
  }
  if (dev >= kMaxDevices) {
    char buf[128];
    snprintf(buf, sizeof(buf), "device %d is beyond the %d devices this entry point keeps scratch addresses for",
             dev, kMaxDevices);
    put(msg, len, buf);
    return MUON_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_ctx_get_current) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      put(msg, len, "cuCtxGetCurrent entry point not found");
      return MUON_ERR_CUDA;
    }
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  // Null while this thread has no context yet; the lookup below creates the device's primary context.
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  ScratchSlot& slot = g_scratch_slot[dev];
  if (!slot.addr || !ctx || slot.ctx != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      put(msg, len, "cudaGetSymbolAddress of the scratch array failed");
      return MUON_ERR_CUDA;
    }
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) {
      put(msg, len, "no current CUDA context");
      return MUON_ERR_CUDA;
    }
    slot.addr = p;
    slot.ctx = ctx;
  }
  *out = slot.addr;
  return MUON_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" muon_status muon_normalize_noalloc(const muon_matrix* in, const muon_matrix* out, int count, float eps,
                                              void* stream, char* msg, int msg_len) {
  muon_status st = muon_check_orthogonalize(in, out, count, 0, msg, msg_len);
  if (st != MUON_OK) return st;
  if (!(eps >= 0.0f)) {
    put(msg, msg_len, "eps must be >= 0");
    return MUON_ERR_INVALID;
  }
  if (count > kNoAllocMaxMatrices) {
    put(msg, msg_len, "more than MUON_NOALLOC_MAX_MATRICES matrices");
    return MUON_ERR_INVALID;
  }
  int64_t chunks = 0;
  int live = 0;
  bool in_f32 = false, out_f32 = false;
  for (int j = 0; j < count; ++j) {
    if (in[j].rows == 0 || in[j].cols == 0) continue;
    chunks += (in[j].rows * in[j].cols + kFlatChunk - 1) / kFlatChunk;
    in_f32 = in[j].dtype == MUON_F32;
    out_f32 = out[j].dtype == MUON_F32;
    ++live;
  }
  if (chunks > kNoAllocMaxChunks) {
    put(msg, msg_len, "total size beyond MUON_NOALLOC_MAX_ELEMENTS (counted in whole 8192-element blocks per matrix)");
    return MUON_ERR_INVALID;
  }
  if (live == 0) return MUON_OK;

  void* base = nullptr;
  if ((st = scratch_for_current_device(&base, msg, msg_len)) != MUON_OK) return st;
  float* partial = static_cast<float*>(base);
  int* tickets = reinterpret_cast<int*>(static_cast<unsigned char*>(base) + kPartialBytes);
  float* inv = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kPartialBytes + kTicketBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The tickets must start at zero; an earlier call leaves them at zero, but clear them anyway.
  cudaError_t e = cudaMemsetAsync(tickets, 0, kTicketBytes, s);
  if (e != cudaSuccess) {
    put(msg, msg_len, cudaGetErrorString(e));
    return MUON_ERR_CUDA;
  }

  MomArgs na;
  MapArgs ma;
  memset(&na, 0, sizeof(na));
  memset(&ma, 0, sizeof(ma));
  na.eps = eps;
  ma.keep = 1.0f;
  int nblocks = 0, mblocks = 0;
  int64_t part_off = 0;
  for (int j = 0; j < count; ++j) {
    if (in[j].rows == 0 || in[j].cols == 0) continue;
    const int k = na.count;
    const int64_t elems = in[j].rows * in[j].cols;
    const int nch = static_cast<int>((elems + kFlatChunk - 1) / kFlatChunk);
    MomMat& N = na.m[k];
    N.g = in[j].ptr;
    N.ld_g = in[j].ld;
    N.rows = static_cast<int>(in[j].rows);
    N.cols = static_cast<int>(in[j].cols);
    N.vec_ok = (in[j].cols % 8 == 0 && in[j].ld == in[j].cols && aligned16(in[j].ptr)) ? 1 : 0;
    N.block_begin = nblocks;
    N.nchunks = nch;
    N.partial = partial + part_off;
    N.ticket = tickets + k;
    N.inv = inv + k;
    nblocks += nch;
    part_off += nch;
    ++na.count;

    MapMat& M = ma.m[k];
    M.src = in[j].ptr;
    M.dst = out[j].ptr;
    M.ld_src = in[j].ld;
    M.ld_dst = out[j].ld;
    M.sr = static_cast<int>(in[j].rows);
    M.sc = static_cast<int>(in[j].cols);
    M.transposed = 0;
    M.vec_ok = (M.sc % 8 == 0 && M.ld_src == M.sc && M.ld_dst == M.sc && aligned16(M.src) && aligned16(M.dst))
                   ? 1 : 0;
    M.block_begin = mblocks;
    M.inv = inv + k;
    mblocks += nch;
    ++ma.count;
  }

  if (in_f32)
    momentum_norm_kernel<false, true><<<nblocks, kEwThreads, 0, s>>>(na);
  else
    momentum_norm_kernel<false, false><<<nblocks, kEwThreads, 0, s>>>(na);
  if (in_f32 && out_f32)
    map_kernel<kScale, true, true><<<mblocks, kEwThreads, 0, s>>>(ma);
  else if (in_f32)
    map_kernel<kScale, true, false><<<mblocks, kEwThreads, 0, s>>>(ma);
  else if (out_f32)
    map_kernel<kScale, false, true><<<mblocks, kEwThreads, 0, s>>>(ma);
  else
    map_kernel<kScale, false, false><<<mblocks, kEwThreads, 0, s>>>(ma);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    put(msg, msg_len, cudaGetErrorString(e));
    return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
