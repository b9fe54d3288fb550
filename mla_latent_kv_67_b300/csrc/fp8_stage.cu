// FP8 latent cache on the tensor cores: mla_decode_attn_fp8_staged.
//
// The cache stays in the FP8 row format of include/mla_b300.h (E4M3 codes of
// c_KV with one float scale per row, k_R in bf16; DeepSeek-V2 MLA page 5.1
// item 3 names quantisation as a further saving). A pass on the CUDA cores
// widens the pages a batch reads into bf16 rows in the caller's workspace
// (code * scale, rounded to bf16; k_R copied), in the batch's own page order
// under an identity block table, and the bf16 decode (the tcgen05 kernel
// wherever it supports the shape) then runs on those rows with its usual plan
// and merge. The cache at rest is 0.57 of
// the bf16 cache; the decode moves the FP8 bytes plus a bf16 write and read
// of the pages the batch touches.
#include <cuda_fp8.h>
#include <stdio.h>

#include "common.cuh"
#include "launch.h"
#include "tc_decode.h"

namespace mla {
namespace fp8s {

// One CTA per (query row b, page p < the row's pages). 256 threads; thread t
// widens 16-byte groups of codes of the page's rows. The identity table entry
// [b][p] = b * max_pages + p is written for every p by the CTAs of p's row.
__global__ void __launch_bounds__(256) widen_pages_kernel(
    const uint8_t* __restrict__ cache, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ seq_lens, int max_pages, int num_pages, int page_size, int d_c,
    int d_r, __nv_bfloat16* __restrict__ stage, int32_t* __restrict__ ident,
    int32_t* dev_status) {
  const int b = blockIdx.y, p = blockIdx.x;
  if (threadIdx.x == 0) ident[(size_t)b * max_pages + p] = b * max_pages + p;
  const int len = seq_lens[b];
  if (len < 1 || (long long)len > (long long)max_pages * page_size) return;  // reported by the plan
  if (p >= (len + page_size - 1) / page_size) return;
  const int rb = MLA_FP8_ROW_BYTES(d_c, d_r), W = d_c + d_r;
  int blk = block_table[(size_t)b * max_pages + p];
  const bool bad = blk < 0 || blk >= num_pages;
  if (bad) {
    if (threadIdx.x == 0) report(dev_status, MLA_DEV_BAD_BLOCK);
    blk = 0;
  }
  __nv_bfloat16* dst0 = stage + ((size_t)b * max_pages + p) * page_size * W;
  const uint8_t* src0 = cache + (size_t)blk * page_size * rb;
  // latent part: 16 codes per item
  const int g_per_row = d_c / 16;
  for (int i = threadIdx.x; i < page_size * g_per_row; i += blockDim.x) {
    const int r = i / g_per_row, gq = i % g_per_row;
    const uint8_t* row = src0 + (size_t)r * rb;
    const float s = *reinterpret_cast<const float*>(row + d_c + 2 * d_r);
    const uint4 codes = *reinterpret_cast<const uint4*>(row + 16 * gq);
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
    uint32_t out[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        __nv_fp8_e4m3 a, c;
        a.__x = (uint8_t)(w[k] >> (16 * hh));
        c.__x = (uint8_t)(w[k] >> (16 * hh + 8));
        const __nv_bfloat162 v = __floats2bfloat162_rn(bad ? 0.f : static_cast<float>(a) * s,
                                                       bad ? 0.f : static_cast<float>(c) * s);
        out[2 * k + hh] = *reinterpret_cast<const uint32_t*>(&v);
      }
    }
    uint4* d = reinterpret_cast<uint4*>(dst0 + (size_t)r * W + 16 * gq);
    d[0] = make_uint4(out[0], out[1], out[2], out[3]);
    d[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
  // RoPE part: bf16 copied, 8 values per item
  const int k_per_row = d_r / 8;
  for (int i = threadIdx.x; i < page_size * k_per_row; i += blockDim.x) {
    const int r = i / k_per_row, q = i % k_per_row;
    const uint4 v = bad ? make_uint4(0u, 0u, 0u, 0u)
                        : reinterpret_cast<const uint4*>(src0 + (size_t)r * rb + d_c)[q];
    reinterpret_cast<uint4*>(dst0 + (size_t)r * W + d_c)[q] = v;
  }
}

}  // namespace fp8s

// Workspace: [decode workspace of the bf16 path][identity table][bf16 rows]
struct Fp8StageLayout {
  size_t ident, stage, total;
};
static Fp8StageLayout fp8_stage_layout(size_t ws_decode, int B, int max_pages, const mla_dims* d) {
  Fp8StageLayout L;
  size_t off = align_up(ws_decode, 256);
  L.ident = off;
  off = align_up(off + sizeof(int32_t) * (size_t)B * max_pages, 256);
  L.stage = off;
  off += (size_t)B * max_pages * d->page_size * (size_t)(d->d_c + d->d_r) * 2;
  L.total = off;
  return L;
}

}  // namespace mla

extern "C" size_t mla_decode_fp8_staged_workspace_size(int B, int max_pages,
                                                       const mla_dims* dims) {
  using namespace mla;
  if (B <= 0 || max_pages <= 0 || check_dims(dims) != MLA_OK) return 0;
  const size_t wsd = mla_decode_workspace_size(B, MLA_BF16, dims);
  if (wsd == 0) return 0;
  return fp8_stage_layout(wsd, B, max_pages, dims).total;
}

extern "C" mla_status mla_decode_attn_fp8_staged(const void* q_cat, const void* cache,
                                                 const int32_t* block_table, int max_pages,
                                                 int num_pages, const int32_t* seq_lens, int B,
                                                 float softmax_scale, void* workspace,
                                                 size_t ws_bytes, float* o_lat, float* lse,
                                                 const mla_dims* d, int32_t* dev_status,
                                                 void* stream) {
  using namespace mla;
  // the bf16 decode's checks and plan layout, on the widened rows
  DecodeSetup ds;
  mla_status st = decode_setup(q_cat, cache, block_table, max_pages, num_pages, seq_lens, B, 1,
                               o_lat, lse, MLA_BF16, d, &ds);
  if (st != MLA_OK || B == 0) return st;
  if (B > 65535 || d->d_r % 8 != 0)
    return record_error(MLA_ERR_UNSUPPORTED, "mla_decode_attn_fp8_staged needs B <= 65535 "
                                             "and d_r a multiple of 8");
  const Fp8StageLayout FL = fp8_stage_layout(ds.L.total, B, max_pages, d);
  if (!workspace || ws_bytes < FL.total) {
    char buf[200];
    snprintf(buf, sizeof(buf), "workspace %zu bytes < %zu required", ws_bytes, FL.total);
    return record_error(MLA_ERR_WORKSPACE, buf);
  }
  if ((reinterpret_cast<uintptr_t>(cache) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return record_error(MLA_ERR_INVALID_ARG,
                        "cache must be 16-byte and workspace 256-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = reinterpret_cast<char*>(workspace);
  auto* stage = reinterpret_cast<__nv_bfloat16*>(ws + FL.stage);
  auto* ident = reinterpret_cast<int32_t*>(ws + FL.ident);
  fp8s::widen_pages_kernel<<<dim3(max_pages, B), 256, 0, s>>>(
      reinterpret_cast<const uint8_t*>(cache), block_table, seq_lens, max_pages, num_pages,
      d->page_size, d->d_c, d->d_r, stage, ident, dev_status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = launch_plan(seq_lens, B, 1, max_pages * (d->page_size / ds.unit), ds.unit, ds.workers,
                    ds.path, true, workspace, ds.L, dev_status, s);
  if (e == cudaSuccess)
    e = launch_decode(ds, q_cat, stage, ident, max_pages, B * max_pages, B, softmax_scale,
                      workspace, o_lat, lse, MLA_BF16, d, dev_status, s);
  if (e == cudaSuccess) e = launch_combine(workspace, ds.L, B, d->n_h, d->d_c, o_lat, lse, s);
  if (e != cudaSuccess) {
    char buf[200];
    snprintf(buf, sizeof(buf), "decode_attn_fp8_staged: %s", cudaGetErrorString(e));
    return record_error(MLA_ERR_CUDA, buf);
  }
  return MLA_OK;
}
