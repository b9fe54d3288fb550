// Allocation-free decode: mla_decode_attn_static.
//
// Some callers cannot allocate device memory at the point where they decode:
// plugin hosts and embedded runtimes that hand a plugin a stream but no
// allocator, and serving loops that forbid device allocations after
// start-up so that no step ever blocks on the allocator. Such a caller has
// no way to provide the decode workspace. This entry point instead keeps
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
  // the same checks, kernel choice and plan layout as mla_decode_attn
  DecodeSetup ds;
  mla_status st = decode_setup(q_cat, cache, block_table, max_pages, num_pages, seq_lens, B, 1,
                               o_lat, lse, dtype, d, &ds);
  if (st != MLA_OK || B == 0) return st;
  if (ds.L.total > (size_t)MLA_STATIC_SCRATCH_BYTES)
    return err(MLA_ERR_WORKSPACE,
               "this batch needs %zu bytes of decode scratch (B=%d, %d workers, n_h=%d, d_c=%d) "
               "but the static scratch holds %zu; use mla_decode_attn with a caller workspace",
               ds.L.total, B, ds.workers, d->n_h, d->d_c, (size_t)MLA_STATIC_SCRATCH_BYTES);
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess)
    return err(MLA_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Nothing in the scratch needs to start at zero: the plan kernel rewrites
  // every plan entry it reads back, and each partial slot is written by the
  // decode kernel before the combine kernel reads it.
  e = launch_plan(seq_lens, B, 1, max_pages * (d->page_size / ds.unit), ds.unit, ds.workers, ds.path,
                  dtype != MLA_F32,
                  ws, ds.L, dev_status, s);
  if (e == cudaSuccess)
    e = launch_decode(ds, q_cat, cache, block_table, max_pages, num_pages, B, softmax_scale, ws,
                      o_lat, lse, dtype, d, dev_status, s);
  if (e == cudaSuccess) e = launch_combine(ws, ds.L, B, d->n_h, d->d_c, o_lat, lse, s);
  if (e != cudaSuccess) return err(MLA_ERR_CUDA, "decode_attn_static: %s", cudaGetErrorString(e));
  return MLA_OK;
}
