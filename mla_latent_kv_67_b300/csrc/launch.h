// Host-side launchers shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mla {

// Generic CUDA-core batched GEMM with fused epilogues:
//   out[g][m][n] = sum_k A[g][m][k] * W[g](n, k)
// A element (g,m,k) at a + g*a_gs + m*a_ms + k*a_ks (a_ks == 0 means 1);
// W element (g,n,k) at w + g*w_gs + n*w_ns + k*w_ks.
enum Epilogue {
  EPI_STORE = 0,   // out + g*o_gs + m*o_ms + n
  EPI_ROPE = 1,    // as STORE, RoPE on columns n%(rope_off+d_r) >= rope_off
  EPI_APPEND = 2,  // RoPE on n >= rope_off, then scatter into the paged cache
};

struct GemmArgs {
  const void* a; long long a_gs, a_ms; int a_f32; long long a_ks;
  const void* w; long long w_gs, w_ns, w_ks; int w_f32;
  int G, M, N, K;
  int epi;
  void* out; long long o_gs, o_ms; int o_f32;
  // RoPE (EPI_ROPE / EPI_APPEND)
  const float* rope; int max_pos; int d_r; int rope_off; int rope_period;
  const int32_t* pos;
  // paged store (EPI_APPEND)
  const int32_t* seq_idx; const int32_t* block_table; int B, max_pages, num_pages, page_size;
  int32_t* dev_status;
};

cudaError_t launch_simt_gemm(const GemmArgs& g, cudaStream_t s);
// tcgen05 weight-streaming version of the same product for G == 1, bf16 A
// and W, W K-major (w_ks == 1), K % 64 == 0 (tc_gemm.cu). `ldx` is A's row
// stride in elements.
bool tc_gemm_supported(int M, int N, int K, long long ldx);
cudaError_t tc_gemm_launch(const GemmArgs& g, long long ldx, cudaStream_t s);
// tcgen05 tile GEMM for many tokens (tc_tgemm.cu): the same products and
// epilogues, tiles of 128 tokens x 256 features, tensor-core bound. Taken
// where tc_tgemm_wanted holds and tc_gemm_supported does.
bool tc_tgemm_wanted(int M, int N, int K);
cudaError_t tc_tgemm_launch(const GemmArgs& g, long long ldx, cudaStream_t s);
cudaError_t launch_copy_rope_part(const void* q, void* q_cat, int B, int n_h, int d_h, int d_r,
                                  int d_c, int f32, cudaStream_t s);
cudaError_t launch_rope_table(float* cs, int max_pos, int d_r, double base, cudaStream_t s);
// dst[g][r][j] = src[g][r][j] for r < rows, j < cols (bf16 or fp32 elements of
// `esz` bytes); row strides in elements, group strides in elements.
cudaError_t launch_copy_rows(const void* src, long long src_gs, long long src_rs, void* dst,
                             long long dst_gs, long long dst_rs, int G, int rows, int cols,
                             int esz, cudaStream_t s);
// rows[t] = the cache row of position t of sequence `seq`, t < n (block ids
// outside the pool are reported and give a zero row).
cudaError_t launch_gather_rows(const void* cache, const int32_t* block_table, int max_pages,
                               int num_pages, int page_size, int seq, int n, int width, int esz,
                               void* rows, int32_t* dev_status, cudaStream_t s);
// dst[i] = bf16(src[i]) for i < n.
cudaError_t launch_to_bf16(const float* src, void* dst, long long n, cudaStream_t s);

// Decode launchers take B = the number of query rows (sequences x new
// tokens per sequence) and bt_div = new tokens per sequence: query row s
// reads block-table row s / bt_div.
cudaError_t launch_simt_decode(const void* q_cat, const void* cache, const int32_t* block_table,
                               int max_pages, int num_pages, int B, int workers, float scale,
                               const void* ws, const WorkspaceLayout& L, float* o_lat, float* lse,
                               int n_h, int d_c, int d_r, int page_size, int unit, int f32,
                               int32_t* dev_status, int bt_div, cudaStream_t s);
// (f32: 1 = fp32 cache and queries, 0 = bf16, 2 = the FP8 row format with
// bf16 queries.)

// Plan for B sequences with q_len new tokens each: B * q_len query rows;
// row v = b * q_len + t sees seq_lens[b] - (q_len - 1 - t) cached tokens.
// part_bf16: the decode kernels keep split partials in bf16 (bf16 and FP8
// caches) rather than fp32 (fp32 cache); the combine reads it from the plan.
cudaError_t launch_plan(const int32_t* seq_lens, int B, int q_len, int max_pages, int page_size,
                        int workers, int path, bool part_bf16, void* ws, const WorkspaceLayout& L,
                        int32_t* dev_status, cudaStream_t s);
cudaError_t launch_combine(const void* ws, const WorkspaceLayout& L, int B, int n_h, int d_c,
                           float* o_lat, float* lse, cudaStream_t s);

mla_status record_error(mla_status st, const char* msg);

// Host-side checks and dispatch shared by the decode entry points (api.cu).
mla_status check_dims(const mla_dims* d);
mla_status check_dtype(int dt);         // MLA_F32 or MLA_BF16
mla_status check_decode_dtype(int dt);  // also MLA_FP8_E4M3 (the FP8 cache)
int pick_path(mla_dtype dt, const mla_dims* d);  // 1 tcgen05, 0 SIMT
int workers_for(int path);                       // workers the plan cuts the pages into
struct DecodeSetup {
  int path, workers;
  int q_len;        // new tokens per sequence (query rows = B * q_len)
  int unit;         // tokens per plan unit (plan_unit)
  WorkspaceLayout L;
};
// Tokens per unit of the split plan: the page, except on the CUDA-core path
// when the batch's pages cannot give every worker one (then 32 tokens, the
// kernel's token tile, so a short batch still spreads over the SMs). The
// plan and the decode call derive it from the same arguments.
int plan_unit(int path, int rows, int max_pages, int page_size, int workers);
// Validates the arguments of a decode call exactly as mla_decode_attn does
// and picks its kernel, worker count and workspace layout. B == 0 is valid
// (nothing to do; `out` then has workers == 0).
mla_status decode_setup(const void* q_cat, const void* cache, const int32_t* block_table,
                        int max_pages, int num_pages, const int32_t* seq_lens, int B, int q_len,
                        const float* o_lat, const float* lse, mla_dtype dtype,
                        const mla_dims* dims, DecodeSetup* out);
// The decode kernel `ds` selects, on workspace `ws` (planned by launch_plan).
cudaError_t launch_decode(const DecodeSetup& ds, const void* q_cat, const void* cache,
                          const int32_t* block_table, int max_pages, int num_pages, int B,
                          float softmax_scale, void* ws, float* o_lat, float* lse, mla_dtype dtype,
                          const mla_dims* d, int32_t* dev_status, cudaStream_t s);

// Raises a kernel's dynamic shared-memory limit once per device, so later
// launches (including ones recorded into a CUDA graph) make no further host
// API call for it. `done` is the caller's per-kernel bit mask of devices.
inline cudaError_t set_max_smem_once(const void* kernel, int bytes, unsigned long long& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && ((done >> dev) & 1ull)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done |= 1ull << dev;
  return e;
}

}  // namespace mla
