// asv_static_scratch.cu -- asymspec_verify_static: the AsymSpec verification for callers that
// cannot allocate device memory themselves.
//
// Some callers are handed only their input and output buffers: a plugin running inside a
// serving framework whose memory pool it does not own, or code that must not allocate once it
// is running (an allocation can block, fragment a pool or fail under memory pressure).  They
// cannot provide the few kilobytes of workspace that asymspec_verify takes (the per-request
// tickets and per-row records of the last-arriver scan).  This entry point keeps that scratch in
// a file-scope device array instead, reserved when the library's device code is loaded on a GPU
// and held by that GPU until the process exits.  It calls no cudaMalloc/cudaFree and no
// allocating library routine.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "asv.h"
#include "asv_internal.h"

namespace {

// The scratch: tickets (one per request, padded to 256 bytes) then one 16-byte record per row.
static __device__ __align__(256) unsigned char g_static_scratch[ASV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up with the device current.  A call made
// outside stream capture looks it up again every time (a device reset reloads the module, and
// the array may then sit at another address); a call made while `stream` is capturing uses the
// address the last call outside capture found on this device (a lookup may load the module,
// which capture does not allow), and looks it up only if there is none yet.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  bool capturing = true;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess) capturing = cs != cudaStreamCaptureStatusNone;
  else cudaGetLastError();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!capturing || !g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" asv_status asymspec_verify_static(const void* a, const void* b, const void* t, int dtype,
                                             const int32_t* draft_ids, int B, int K, int V, float beta, float gamma,
                                             int32_t* out_accept_len, int32_t* out_tokens, float* out_D,
                                             float* out_lse, uint32_t* out_req_status, cudaStream_t stream) {
  // Every check comes before the GPU or the shared array is touched: shapes (with the overflow
  // guard on B * (K + 1)) first, so that the workspace size is computed only for a valid shape;
  // then the size limit; then the checks asymspec_verify applies to its arguments.
  asv_status st = asv::check_asym_shape(B, K, V, dtype);
  if (st != ASV_OK) return st;
  // The scratch serves the cluster kernel (tickets and row records only): the call passes exactly
  // that much, which keeps the staged kernel's exchange area, and the counters in it that would
  // have to start at zero, out of the shared array.
  const size_t need = asv::asym_cluster_workspace_bytes(B, K);
  if (need > size_t(ASV_STATIC_SCRATCH_BYTES)) return ASV_ERR_WORKSPACE;  // batch too large for the static scratch
  if (B == 0) return ASV_OK;
  st = asv::check_asym_args(a, b, t, dtype, draft_ids, K, beta, gamma, out_accept_len, out_tokens, out_D, out_lse,
                            out_req_status);
  if (st != ASV_OK) return st;
  void* ws = nullptr;
  cudaError_t e = scratch_address(stream, &ws);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ASV_ERR_CUDA;
  }
  // The scan's tickets must start at zero.  A finished call leaves them zero, but the array is
  // shared by every call, so clear them on the stream rather than trust what the last call left.
  const size_t tickets = (size_t(B) * 4 + 255) / 256 * 256;
  e = cudaMemsetAsync(ws, 0, tickets, stream);
  if (e != cudaSuccess) return ASV_ERR_CUDA;
  return asymspec_verify(a, b, t, dtype, draft_ids, B, K, V, beta, gamma, out_accept_len, out_tokens, out_D, out_lse,
                         out_req_status, ws, need, stream);
}
