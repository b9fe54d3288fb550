// Allocation-free decode: mla_decode_attn_static.
//
// Some callers cannot allocate device memory at the point where they decode:
// code running under a CUDA stream capture in global mode (cudaMalloc is not
// permitted there), plugin hosts and embedded runtimes that hand a plugin a
// stream but no allocator, and serving loops that forbid driver allocations
// after start-up so that no step ever blocks on the allocator. Such a caller
// has no way to provide the decode workspace. This entry point instead keeps
// that workspace (split plan plus split-KV partial results) in one
// file-scope device array of fixed size, so the call itself allocates
// nothing; the caller still provides every input and output tensor.
#include <mutex>
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"
#include "launch.h"
#include "tc_decode.h"

namespace {

// The static scratch: every GPU that loads this library holds it until the
// process exits. Calls share it, so two calls that overlap on the GPU (other
// streams, or other host threads) race on its contents.
static __device__ __align__(256) unsigned char g_static_scratch[MLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device. In host code `g_static_scratch` names a host-side stand-in, never
// the device array, so it must not be handed to a kernel.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

mla_status err(mla_status st, const char* fmt, ...) {
  char buf[400];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  return mla::record_error(st, buf);
}

}  // namespace

extern "C" mla_status mla_decode_attn_static(const void* q_cat, const void* cache,
                                             const int32_t* block_table, int max_pages,
                                             int num_pages, const int32_t* seq_lens, int B,
                                             float softmax_scale, float* o_lat, float* lse,
                                             mla_dtype dtype, const mla_dims* d,
                                             int32_t* dev_status, void* stream) {
  using namespace mla;
  if (!d) return err(MLA_ERR_INVALID_ARG, "dims is NULL");
  if (dtype != MLA_F32 && dtype != MLA_BF16) return err(MLA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (d->n_h <= 0 || d->d_c <= 0 || d->d_h <= 0 || d->d_v <= 0 || d->page_size <= 0 ||
      d->d_r < 0 || d->d_r % 2)
    return err(MLA_ERR_INVALID_ARG, "bad dims");
  if (B < 0) return err(MLA_ERR_INVALID_ARG, "B must be >= 0");
  if (B == 0) return MLA_OK;
  if (!q_cat || !cache || !block_table || !seq_lens || !o_lat || !lse)
    return err(MLA_ERR_INVALID_ARG, "NULL tensor argument");
  if (max_pages <= 0 || num_pages <= 0)
    return err(MLA_ERR_INVALID_ARG, "max_pages and num_pages must be > 0");
  if (d->d_c % 32 != 0 || d->d_c > 512)
    return err(MLA_ERR_INVALID_ARG, "d_c must be a multiple of 32, <= 512");
  const int path = mla_decode_path(dtype, d);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return err(MLA_ERR_CUDA, "cannot query the device's SM count");
  const int workers = path == 1 ? tc_pair_workers(sms) : sms;
  const WorkspaceLayout L = workspace_layout(B, workers, d->n_h, d->d_c);
  if (L.total > (size_t)MLA_STATIC_SCRATCH_BYTES)
    return err(MLA_ERR_WORKSPACE,
               "this batch needs %zu bytes of decode scratch (B=%d, %d workers, n_h=%d, d_c=%d) "
               "but the static scratch holds %zu; use mla_decode_attn with a caller workspace",
               L.total, B, workers, d->n_h, d->d_c, (size_t)MLA_STATIC_SCRATCH_BYTES);
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess)
    return err(MLA_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Nothing in the scratch needs to start at zero: the plan kernel rewrites
  // every plan entry it reads back, and each partial slot is written by the
  // decode kernel before the combine kernel reads it.
  e = launch_plan(seq_lens, B, max_pages, d->page_size, workers, path, ws, L, dev_status, s);
  if (e == cudaSuccess) {
    if (path == 1)
      e = tc_pair_launch(q_cat, cache, block_table, max_pages, num_pages, B, workers,
                         softmax_scale, ws, L, o_lat, lse, dev_status, s);
    else
      e = launch_simt_decode(q_cat, cache, block_table, max_pages, num_pages, B, workers,
                             softmax_scale, ws, L, o_lat, lse, d->n_h, d->d_c, d->d_r,
                             d->page_size, dtype == MLA_F32, dev_status, s);
  }
  if (e == cudaSuccess) e = launch_combine(ws, L, B, d->n_h, d->d_c, o_lat, lse, s);
  if (e != cudaSuccess) return err(MLA_ERR_CUDA, "decode_attn_static: %s", cudaGetErrorString(e));
  return MLA_OK;
}
