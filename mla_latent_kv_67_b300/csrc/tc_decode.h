// tcgen05 (5th-generation tensor core) decode attention: host interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mla {

// Shapes the tensor-core kernel is built for (DeepSeek-V2 MLA: 128 heads,
// 512-wide latent, 64-wide RoPE key, 64-token pages).
bool tc_decode_supported(int n_h, int d_c, int d_r, int page_size);
// Test build only (MLA_TEST_HOOKS): when set, the tensor-core decode
// kernels' page producers issue nothing, so their bounded waits run out.
extern int g_test_withhold;
// The latent-split pair kernel (each CTA of a cluster owns half of d_c).
int tc_split_workers(int sms);
cudaError_t tc_split_launch(const void* q_cat, const void* cache, const int32_t* block_table,
                            int max_pages, int num_pages, int B, int workers, float scale,
                            const void* ws, const WorkspaceLayout& L, float* o_lat, float* lse,
                            int32_t* dev_status, int bt_div, cudaStream_t s);
// The score/value pair kernel (score CTA + value CTA per worker).
int tc_pair_workers(int sms);
cudaError_t tc_pair_launch(const void* q_cat, const void* cache, const int32_t* block_table,
                           int max_pages, int num_pages, int B, int workers, float scale,
                           const void* ws, const WorkspaceLayout& L, float* o_lat, float* lse,
                           int32_t* dev_status, int bt_div, cudaStream_t s);

// tcgen05 absorption products (DeepSeek-V2 shapes, bf16 weights).
bool tc_absorb_supported(int n_h, int d_h, int d_r, int d_c, int d_v);
cudaError_t tc_absorb_q_launch(const void* q, const void* w_uk, void* q_cat, int B,
                               int32_t* dev_status, cudaStream_t s);
cudaError_t tc_absorb_out_launch(const float* o_lat, const void* w_uv, void* o, int out_f32, int B,
                                 int32_t* dev_status, cudaStream_t s);
// mla_combine fused into absorb_out (plan and partials from `ws`).
cudaError_t tc_absorb_out_merge_launch(const void* ws, const WorkspaceLayout& L, float* o_lat,
                                       float* lse, const void* w_uv, void* o, int out_f32, int B,
                                       int32_t* dev_status, cudaStream_t s);

// Causal prefill attention in the MHA form (tc_prefill.cu): DeepSeek-V2
// shapes, bf16. q [N][128][192], k_nope [N][128][128], rows [N][576] (k_R =
// columns 512..575), v [N][128][128] -> o [N][128][128] bf16, lse [N][128].
bool tc_prefill_supported(int n_h, int d_h, int d_r, int d_c, int d_v);
cudaError_t tc_prefill_launch(const void* q, const void* k_nope, const void* rows, const void* v,
                              void* o, float* lse, int N, float scale, int32_t* dev_status,
                              cudaStream_t s);

// One page of the decode's tensor-core data path without softmax:
// s_out[128][64] = q_cat[128][576] . page[64][576]^T and
// o_out[128][256] = pmat[128][64] . page[:, 256 r : 256 r + 256].
cudaError_t tc_selftest_launch(const void* q_cat, const void* page, const void* pmat, float* s_out,
                               float* o_out, int r, int32_t* dev_status, cudaStream_t s);

}  // namespace mla
