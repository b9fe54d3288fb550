// CUDA-core (SIMT) kernels: the generic-shape path.
//
// They serve every dtype/shape the tensor-core kernels do not (the fp32 path,
// small head counts) and give the tensor-core kernels an independent GPU
// cross-check. fp32 arithmetic throughout; bf16 operands are widened on load.
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace mla {

// ------------------------------------------------------------- RoPE table
__global__ void rope_table_kernel(float* cs, int max_pos, int half, double base, int d_r) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)max_pos * half) return;
  const int p = (int)(i / half), k = (int)(i % half);
  const double theta = pow(base, -2.0 * (double)k / (double)d_r);
  double sn, cn;
  sincos((double)p * theta, &sn, &cn);
  cs[2 * i] = (float)cn;
  cs[2 * i + 1] = (float)sn;
}

cudaError_t launch_rope_table(float* cs, int max_pos, int d_r, double base, cudaStream_t s) {
  const long long n = (long long)max_pos * (d_r / 2);
  if (n == 0) return cudaSuccess;
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(cs, max_pos, d_r / 2, base, d_r);
  return cudaGetLastError();
}

// ------------------------------------------------------------ batched GEMM
constexpr int GB_M = 32, GB_N = 64, GB_K = 32;

__device__ __forceinline__ float ld_any(const void* p, long long i, int f32) {
  return f32 ? reinterpret_cast<const float*>(p)[i]
             : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}
__device__ __forceinline__ void st_any(void* p, long long i, float v, int f32) {
  if (f32) reinterpret_cast<float*>(p)[i] = v;
  else reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// 256 threads; thread (tx, ty) computes columns n0+2tx, n0+2tx+1 of rows
// m0+ty+8i, i < 4, so a RoPE pair (2i, 2i+1) never straddles threads.
__global__ void __launch_bounds__(256) simt_gemm_kernel(GemmArgs p) {
  __shared__ float As[GB_M][GB_K + 1];
  __shared__ float Ws[GB_K][GB_N + 1];
  const int g = blockIdx.z;
  const int m0 = blockIdx.y * GB_M, n0 = blockIdx.x * GB_N;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const long long a_base = (long long)g * p.a_gs;
  const long long a_ks = p.a_ks ? p.a_ks : 1;
  const long long w_base = (long long)g * p.w_gs;
  const bool w_kmajor = p.w_ks == 1;
  float acc[4][2] = {};
  for (int k0 = 0; k0 < p.K; k0 += GB_K) {
    for (int idx = threadIdx.x; idx < GB_M * GB_K; idx += 256) {
      const int mm = idx / GB_K, kk = idx % GB_K;
      const int m = m0 + mm, k = k0 + kk;
      As[mm][kk] = (m < p.M && k < p.K) ? ld_any(p.a, a_base + m * p.a_ms + k * a_ks, p.a_f32) : 0.f;
    }
    for (int idx = threadIdx.x; idx < GB_N * GB_K; idx += 256) {
      int nn, kk;
      if (w_kmajor) { nn = idx / GB_K; kk = idx % GB_K; }
      else          { nn = idx % GB_N; kk = idx / GB_N; }
      const int n = n0 + nn, k = k0 + kk;
      Ws[kk][nn] = (n < p.N && k < p.K)
                       ? ld_any(p.w, w_base + (long long)n * p.w_ns + (long long)k * p.w_ks, p.w_f32)
                       : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < GB_K; ++kk) {
      const float w0 = Ws[kk][2 * tx], w1 = Ws[kk][2 * tx + 1];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = As[ty + 8 * i][kk];
        acc[i][0] = fmaf(a, w0, acc[i][0]);
        acc[i][1] = fmaf(a, w1, acc[i][1]);
      }
    }
    __syncthreads();
  }
  const int n = n0 + 2 * tx;
  if (n >= p.N) return;
  const bool pair = n + 1 < p.N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 8 * i;
    if (m >= p.M) continue;
    float v0 = acc[i][0], v1 = acc[i][1];
    if (p.epi == EPI_ROPE || p.epi == EPI_APPEND) {
      const int col = p.epi == EPI_ROPE ? n % p.rope_period : n;
      if (col >= p.rope_off && pair) {
        const int ps = p.pos[m];
        if (ps < 0 || ps >= p.max_pos) {
          report(p.dev_status, MLA_DEV_BAD_POS);
        } else {
          const int k = (col - p.rope_off) >> 1;
          const float c = p.rope[((size_t)ps * (p.d_r / 2) + k) * 2];
          const float s = p.rope[((size_t)ps * (p.d_r / 2) + k) * 2 + 1];
          const float e = v0, o = v1;
          v0 = e * c - o * s;
          v1 = e * s + o * c;
        }
      }
    }
    if (p.epi == EPI_APPEND) {
      const int sq = p.seq_idx ? p.seq_idx[m] : m;
      const int ps = p.pos[m];
      if (sq < 0 || sq >= p.B || ps < 0 || ps >= p.max_pages * p.page_size) {
        report(p.dev_status, MLA_DEV_BAD_POS);
        continue;
      }
      const int blk = p.block_table[(size_t)sq * p.max_pages + ps / p.page_size];
      if (blk < 0 || blk >= p.num_pages) {
        report(p.dev_status, MLA_DEV_BAD_BLOCK);
        continue;
      }
      const long long row = (long long)blk * p.page_size + ps % p.page_size;
      st_any(p.out, row * p.N + n, v0, p.o_f32);
      if (pair) st_any(p.out, row * p.N + n + 1, v1, p.o_f32);
    } else {
      const long long o = (long long)g * p.o_gs + (long long)m * p.o_ms + n;
      st_any(p.out, o, v0, p.o_f32);
      if (pair) st_any(p.out, o + 1, v1, p.o_f32);
    }
  }
}

cudaError_t launch_simt_gemm(const GemmArgs& g, cudaStream_t s) {
  if (g.M == 0 || g.N == 0 || g.G == 0) return cudaSuccess;
  dim3 grid((g.N + GB_N - 1) / GB_N, (g.M + GB_M - 1) / GB_M, g.G);
  simt_gemm_kernel<<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

__global__ void copy_rows_kernel(const char* src, long long src_gs, long long src_rs, char* dst,
                                 long long dst_gs, long long dst_rs, int rows, int cols, int esz) {
  const int g = blockIdx.y;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)rows * cols;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / cols, j = i % cols;
    const char* a = src + (g * src_gs + r * src_rs + j) * esz;
    char* b = dst + (g * dst_gs + r * dst_rs + j) * esz;
    if (esz == 4) *reinterpret_cast<float*>(b) = *reinterpret_cast<const float*>(a);
    else *reinterpret_cast<__nv_bfloat16*>(b) = *reinterpret_cast<const __nv_bfloat16*>(a);
  }
}

cudaError_t launch_copy_rows(const void* src, long long src_gs, long long src_rs, void* dst,
                             long long dst_gs, long long dst_rs, int G, int rows, int cols,
                             int esz, cudaStream_t s) {
  if (G == 0 || rows == 0 || cols == 0) return cudaSuccess;
  const long long n = (long long)rows * cols;
  const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  copy_rows_kernel<<<dim3(blocks, G), 256, 0, s>>>((const char*)src, src_gs, src_rs, (char*)dst,
                                                   dst_gs, dst_rs, rows, cols, esz);
  return cudaGetLastError();
}

__global__ void gather_rows_kernel(const uint4* __restrict__ cache, const int32_t* __restrict__ bt,
                                   int max_pages, int num_pages, int page_size, int seq, int n,
                                   int w16, uint4* __restrict__ rows, int32_t* dev_status) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)n * w16;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / w16), u = (int)(i % w16);
    const int blk = bt[(size_t)seq * max_pages + t / page_size];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (blk < 0 || blk >= num_pages) report(dev_status, MLA_DEV_BAD_BLOCK);
    else v = cache[((size_t)blk * page_size + t % page_size) * w16 + u];
    rows[i] = v;
  }
}

cudaError_t launch_gather_rows(const void* cache, const int32_t* block_table, int max_pages,
                               int num_pages, int page_size, int seq, int n, int width, int esz,
                               void* rows, int32_t* dev_status, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if ((width * esz) % 16 != 0) return cudaErrorInvalidValue;
  const int w16 = width * esz / 16;
  const long long total = (long long)n * w16;
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  gather_rows_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(cache), block_table,
                                            max_pages, num_pages, page_size, seq, n, w16,
                                            reinterpret_cast<uint4*>(rows), dev_status);
  return cudaGetLastError();
}

__global__ void to_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    dst[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
}

cudaError_t launch_to_bf16(const float* src, void* dst, long long n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (n % 4 != 0) return cudaErrorInvalidValue;
  const long long n4 = n / 4;
  const int blocks = (int)((n4 + 255) / 256 < 2048 ? (n4 + 255) / 256 : 2048);
  to_bf16_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(src),
                                         reinterpret_cast<uint2*>(dst), n4);
  return cudaGetLastError();
}

// q_cat[b][h][d_c + r] = q[b][h][d_h + r]
__global__ void copy_rope_part_kernel(const void* q, void* q_cat, int B, int n_h, int d_h, int d_r,
                                      int d_c, int f32) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * n_h * d_r) return;
  const long long bh = i / d_r;
  const int r = (int)(i % d_r);
  const long long src = bh * (d_h + d_r) + d_h + r, dst = bh * (d_c + d_r) + d_c + r;
  if (f32) reinterpret_cast<float*>(q_cat)[dst] = reinterpret_cast<const float*>(q)[src];
  else reinterpret_cast<__nv_bfloat16*>(q_cat)[dst] = reinterpret_cast<const __nv_bfloat16*>(q)[src];
}

cudaError_t launch_copy_rope_part(const void* q, void* q_cat, int B, int n_h, int d_h, int d_r,
                                  int d_c, int f32, cudaStream_t s) {
  const long long n = (long long)B * n_h * d_r;
  if (n == 0) return cudaSuccess;
  copy_rope_part_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(q, q_cat, B, n_h, d_h, d_r, d_c, f32);
  return cudaGetLastError();
}

// ------------------------------------------------------------ decode (SIMT)
// Grid (workers, ceil(n_h/8)); 8 warps, one head per warp. Tokens are
// processed 32 at a time: the block stages the 32 cache rows in shared
// memory (fp32, rows padded by one word), lane t scores token t, the warp
// runs the online-softmax update and lane l accumulates latent columns
// l, l+32, ... (d_c <= 512, d_c % 32 == 0).
constexpr int SD_HEADS = 8, SD_TOK = 32, SD_MAXC = 16;

// Cache row readers: element k of physical row `row`, widened to float.
template <typename T>
struct ElemRows {  // [rows][W] of T (float or bf16)
  const T* c;
  int W;
  __device__ float operator()(long long row, int k) const { return load_elem(c, row * W + k); }
};
struct Fp8Rows {  // the FP8 row format of include/mla_b300.h
  const uint8_t* c;
  int rb, d_c, d_r;
  __device__ float operator()(long long row, int k) const {
    const uint8_t* r = c + row * rb;
    if (k < d_c) {
      __nv_fp8_e4m3 v;
      v.__x = r[k];
      return static_cast<float>(v) * *reinterpret_cast<const float*>(r + d_c + 2 * d_r);
    }
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(r + d_c)[k - d_c]);
  }
};

template <typename T, typename Rows>
__global__ void __launch_bounds__(256) simt_decode_kernel(
    const T* __restrict__ q_cat, const Rows cache, const int32_t* __restrict__ block_table,
    int max_pages, int num_pages, int B, float scale, const char* __restrict__ ws, WorkspaceLayout L,
    float* __restrict__ o_lat, float* __restrict__ lse_out, int n_h, int d_c, int d_r,
    int page_size, int unit, int32_t* dev_status, int bt_div) {
  extern __shared__ float smem[];
  const int W = d_c + d_r, Wp = W + 1;
  float* tile = smem;                     // [SD_TOK][Wp]
  float* qs = tile + SD_TOK * Wp;         // [SD_HEADS][W]
  __shared__ long long row_idx[SD_TOK];   // physical row of each staged token, -1 = skip

  const WorkerPlan wp = reinterpret_cast<const WorkerPlan*>(ws + L.workers)[blockIdx.x];
  if (wp.n_pages == 0) return;
  const SeqPlan* seqs = reinterpret_cast<const SeqPlan*>(ws + L.seqs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * SD_HEADS + warp;
  const bool live = h < n_h;
  const int ncol = d_c / 32;

  for (int s = wp.seq_begin; s <= wp.seq_end; ++s) {
    const SeqPlan sp = seqs[s];
    if (sp.pages == 0) continue;
    const int p0 = s == wp.seq_begin ? wp.page_begin : 0;
    const int p1 = s == wp.seq_end ? wp.page_end + 1 : sp.pages;
    if (p0 >= p1) continue;
    const int tok0 = p0 * unit, tok1 = min(p1 * unit, sp.len);  // plan units of `unit` tokens

    __syncthreads();
    for (int i = threadIdx.x; i < SD_HEADS * W; i += blockDim.x) {
      const int hh = blockIdx.y * SD_HEADS + i / W;
      qs[i] = hh < n_h ? load_elem(q_cat, ((size_t)s * n_h + hh) * W + i % W) : 0.f;
    }
    float m = -INFINITY, l = 0.f, acc[SD_MAXC];
#pragma unroll
    for (int i = 0; i < SD_MAXC; ++i) acc[i] = 0.f;

    for (int t0 = tok0; t0 < tok1; t0 += SD_TOK) {
      const int nt = min(SD_TOK, tok1 - t0);
      __syncthreads();
      if (threadIdx.x < SD_TOK) {
        long long ri = -1;
        if ((int)threadIdx.x < nt) {
          const int tok = t0 + threadIdx.x;
          const int blk = block_table[(size_t)(s / bt_div) * max_pages + tok / page_size];
          if (blk < 0 || blk >= num_pages) report(dev_status, MLA_DEV_BAD_BLOCK);
          else ri = (long long)blk * page_size + tok % page_size;
        }
        row_idx[threadIdx.x] = ri;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < nt * W; i += blockDim.x) {
        const int r = i / W, k = i % W;
        const long long ri = row_idx[r];
        tile[r * Wp + k] = ri >= 0 ? cache(ri, k) : 0.f;
      }
      __syncthreads();
      if (live) {
        float sc = -INFINITY;
        if (lane < nt) {
          const float* qh = qs + warp * W;
          const float* row = tile + lane * Wp;
          float a = 0.f;
          for (int k = 0; k < W; ++k) a = fmaf(qh[k], row[k], a);
          sc = a * scale;
        }
        float mt = sc;
        for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        const float m_new = fmaxf(m, mt);
        const float alpha = expf(m - m_new);
        const float p = lane < nt ? expf(sc - m_new) : 0.f;
        float ps = p;
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l = l * alpha + ps;
#pragma unroll
        for (int i = 0; i < SD_MAXC; ++i) acc[i] *= alpha;
        for (int r = 0; r < nt; ++r) {
          const float pr = __shfl_sync(0xffffffffu, p, r);
          const float* row = tile + r * Wp;
#pragma unroll
          for (int i = 0; i < SD_MAXC; ++i)
            if (i < ncol) acc[i] = fmaf(pr, row[lane + 32 * i], acc[i]);
        }
        m = m_new;
      }
    }
    if (live) {
      const float inv = 1.f / l;
      float* lse_dst;
      if (sp.n_splits == 1) {
        float* dst = o_lat + ((size_t)s * n_h + h) * d_c;
        lse_dst = lse_out + (size_t)s * n_h + h;
#pragma unroll
        for (int i = 0; i < SD_MAXC; ++i)
          if (i < ncol) dst[lane + 32 * i] = acc[i] * inv;
      } else {
        // a split partial: bf16 for bf16 / FP8 caches, fp32 for fp32
        const int slot = sp.slot_begin + (blockIdx.x - sp.first_worker);
        const size_t e0 = ((size_t)slot * n_h + h) * d_c;
        char* op = const_cast<char*>(ws) + L.o_part;
        lse_dst = reinterpret_cast<float*>(const_cast<char*>(ws) + L.lse_part) + (size_t)slot * n_h + h;
#pragma unroll
        for (int i = 0; i < SD_MAXC; ++i)
          if (i < ncol) store_elem(reinterpret_cast<T*>(op), e0 + lane + 32 * i, acc[i] * inv);
      }
      if (lane == 0) *lse_dst = m + logf(l);
    }
  }
}

template <typename T, typename Rows>
static cudaError_t simt_decode_launch(const T* q_cat, const Rows& rows, const int32_t* block_table,
                                      int max_pages, int num_pages, int B, int workers, float scale,
                                      const void* ws, const WorkspaceLayout& L, float* o_lat,
                                      float* lse, int n_h, int d_c, int d_r, int page_size,
                                      int unit, int32_t* dev_status, int bt_div, cudaStream_t s) {
  const int W = d_c + d_r;
  const size_t smem = sizeof(float) * ((size_t)SD_TOK * (W + 1) + (size_t)SD_HEADS * W);
  const dim3 grid(workers, (n_h + SD_HEADS - 1) / SD_HEADS);
  cudaError_t e = cudaFuncSetAttribute(simt_decode_kernel<T, Rows>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  simt_decode_kernel<T, Rows><<<grid, 256, smem, s>>>(q_cat, rows, block_table, max_pages,
                                                      num_pages, B, scale, (const char*)ws, L,
                                                      o_lat, lse, n_h, d_c, d_r, page_size, unit,
                                                      dev_status, bt_div);
  return cudaGetLastError();
}

cudaError_t launch_simt_decode(const void* q_cat, const void* cache, const int32_t* block_table,
                               int max_pages, int num_pages, int B, int workers, float scale,
                               const void* ws, const WorkspaceLayout& L, float* o_lat, float* lse,
                               int n_h, int d_c, int d_r, int page_size, int unit, int f32,
                               int32_t* dev_status, int bt_div, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const int W = d_c + d_r;
  if (f32 == 1)
    return simt_decode_launch((const float*)q_cat, ElemRows<float>{(const float*)cache, W},
                              block_table, max_pages, num_pages, B, workers, scale, ws, L, o_lat,
                              lse, n_h, d_c, d_r, page_size, unit, dev_status, bt_div, s);
  if (f32 == 0)
    return simt_decode_launch((const __nv_bfloat16*)q_cat,
                              ElemRows<__nv_bfloat16>{(const __nv_bfloat16*)cache, W}, block_table,
                              max_pages, num_pages, B, workers, scale, ws, L, o_lat, lse, n_h, d_c,
                              d_r, page_size, unit, dev_status, bt_div, s);
  // FP8 latent cache, bf16 queries
  const Fp8Rows rows{(const uint8_t*)cache, MLA_FP8_ROW_BYTES(d_c, d_r), d_c, d_r};
  return simt_decode_launch((const __nv_bfloat16*)q_cat, rows, block_table, max_pages, num_pages,
                            B, workers, scale, ws, L, o_lat, lse, n_h, d_c, d_r, page_size, unit,
                            dev_status, bt_div, s);
}

}  // namespace mla
