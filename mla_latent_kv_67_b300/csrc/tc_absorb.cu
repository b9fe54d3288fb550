// tcgen05 kernels for the two per-head absorption products of decode
// ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现", 2.2: W^UK
// folds into the query, W^UV maps the latent output back; DeepSeek-V2
// shapes: 128 heads, d_h = d_v = 128, d_c = 512, d_R = 64, bf16 weights).
//
// Both are weight-streaming products with a small batch: every head's
// weight block is read once, and the batch is the MMA's N dimension, so each
// CTA computes D[128 x NT] = W-tile . X^T for one head and NT batch rows:
//
//   absorb_q:   q_cat[b, h, c] = sum_k q[b, h, k] W^UK[h*128 + k, c]
//               A = W^UK_h^T (M = 128 latent columns c, K = 128, MN-major,
//               straight from the row-major weight), B = q rows (K-major),
//               one CTA per (128-column tile of c, head, batch tile). The
//               RoPE part q_cat[b, h, 512:576] = q[b, h, 128:192] is copied
//               by the first column tile.
//   absorb_out: o[b, h*128 + v] = sum_c o_lat[b, h, c] W^UV[h*128 + v, c]
//               A = W^UV_h (M = 128, K = 512, K-major), B = o_lat rows. The
//               fp32 latent output is split into bf16 hi + lo parts (x = hi
//               + lo to about 16 significant bits), stacked along N and both
//               multiplied, so the tensor-core product keeps fp32-like input
//               precision.
//
// Weights come in by TMA with 128-byte swizzle; activations by TMA (q) or
// by the threads that split them (o_lat). fp32 accumulation in TMEM; one
// thread issues the MMAs; all four warps run the epilogue (TMEM lane =
// output row). Waits are bounded and report MLA_DEV_TIMEOUT.
#include <cudaTypedefs.h>

#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_decode.h"

namespace mla {
namespace tca {

using namespace ptx;

constexpr int NH = 128, DH = 128, DR = 64, DC = 512, DV = 128;
constexpr int QW = DH + DR;   // q row width (192)
constexpr int QC = DC + DR;   // q_cat row width (576)
constexpr int NT = 32;        // batch rows per CTA
constexpr uint64_t WAIT_NS = 2000000000ull;

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int32_t* st) {
  volatile int dummy = 0;
  return mbar_wait_bounded(bar, parity, &dummy, st, WAIT_NS);
}

// ------------------------------------------------------------- absorb_q
// smem: A0 | A1 (W^UK_h rows k, columns c0..c0+63 / c0+64..c0+127; 16 KB
// each) | B0 | B1 (q rows, k 0..63 / 64..127; NT x 128 B each) | barriers.
constexpr uint32_t AQ_A = 0, AQ_B = 2 * 16384, AQ_BAR = AQ_B + 2 * NT * 128;
constexpr uint32_t AQ_SMEM = AQ_BAR + 64 + 1024;
constexpr uint32_t IDESC_AQ = idesc_bf16_f32(128, NT, true, false);

__global__ void __launch_bounds__(128)
    absorb_q_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                    const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ q_cat, int B,
                    int32_t* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_tma = sb + AQ_BAR, bar_mma = bar_tma + 8;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + AQ_BAR + 16);
  const int mt = blockIdx.x, h = blockIdx.y, b0 = blockIdx.z * NT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_q);
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), 32);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  bool ok = true;
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar_tma, 2 * 16384 + 2 * NT * 128);
    for (int i = 0; i < 2; ++i) {
      tma_load_2d(sb + AQ_A + i * 16384, &tm_w, 128 * mt + 64 * i, DH * h, bar_tma);
      tma_load_3d(sb + AQ_B + i * NT * 128, &tm_q, 64 * i, h, b0, bar_tma);
    }
    ok = wait_bar(bar_tma, 0, dev_status);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk)
        mma_ss(tmem, sdesc_sw128(sb + AQ_A + kk * 2048, 16384, 1024),
               sdesc_sw128(sb + AQ_B + (kk >> 2) * NT * 128 + (kk & 3) * 32, 16, 1024), IDESC_AQ,
               kk > 0 ? 1u : 0u);
    }
    mma_commit(bar_mma);  // also drains on failure (no MMA issued then)
  }
  // RoPE part of q_cat, copied by the first column tile
  if (mt == 0) {
    for (int i = threadIdx.x; i < NT * 8; i += 128) {
      const int r = i >> 3, u = i & 7;
      if (b0 + r < B) {
        const uint4 v = reinterpret_cast<const uint4*>(q + ((size_t)(b0 + r) * NH + h) * QW + DH)[u];
        reinterpret_cast<uint4*>(q_cat + ((size_t)(b0 + r) * NH + h) * QC + DC)[u] = v;
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  const bool done = __all_sync(0xffffffffu, wait_bar(bar_mma, 0, dev_status));  // warp-uniform for tcgen05.ld
  if (ok && done) {
    tc_fence_after();
    uint32_t v[32];
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16), v);
    tmem_ld_wait();
    const int c = 128 * mt + 32 * warp + lane;
#pragma unroll
    for (int j = 0; j < NT; ++j)
      if (b0 + j < B) q_cat[((size_t)(b0 + j) * NH + h) * QC + c] = __float2bfloat16_rn(__uint_as_float(v[j]));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

// ----------------------------------------------------------- absorb_out
// smem: A (W^UV_h, 8 chunks of 128 rows x 128 B = 128 KB, one barrier per
// chunk so the products start while later chunks are in flight) | B (8
// chunks of 2 NT rows x 128 B: rows 0..NT-1 the hi parts of the NT o_lat
// rows, rows NT..2NT-1 their lo parts) | barriers. One N = 2 NT product per
// 16-wide K step gives D = [W.hi^T | W.lo^T]; the epilogue adds the halves.
constexpr int AO_N = 2 * NT;
constexpr uint32_t AO_A = 0, AO_B = 8 * 16384, AO_BAR = AO_B + 8 * AO_N * 128;
constexpr uint32_t AO_SMEM = AO_BAR + 128 + 1024;
constexpr uint32_t IDESC_AO = idesc_bf16_f32(128, AO_N, false, false);

__global__ void __launch_bounds__(128)
    absorb_out_kernel(const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ o_lat,
                      void* __restrict__ o, int out_f32, int B, int32_t* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_tma = sb + AO_BAR, bar_mma = bar_tma + 8 * 8;  // 8 chunk barriers, then MMA
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + AO_BAR + 80);
  const int h = blockIdx.x, b0 = blockIdx.y * NT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    for (int c = 0; c < 9; ++c) mbar_init(bar_tma + 8 * c, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), AO_N);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (threadIdx.x == 0) {
    for (int c = 0; c < 8; ++c) {
      mbar_expect_tx(bar_tma + 8 * c, 16384);
      tma_load_2d(sb + AO_A + c * 16384, &tm_w, 64 * c, DV * h, bar_tma + 8 * c);
    }
  }
  // B: warp w splits o_lat rows 8w .. 8w + 7 into bf16 hi (tile row r) and
  // lo (tile row NT + r) parts, written in the 128-byte-swizzled K-major
  // layout. Lane l holds float4 columns l, l + 32, l + 64, l + 96 of a row,
  // so each load instruction reads 512 contiguous bytes; all 32 loads of a
  // thread are in flight together (rows past the batch read the last row and
  // are zeroed afterwards).
  {
    float4 x[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 8 * warp + i;
      const int rb = b0 + r < B ? b0 + r : B - 1;
      const float4* src = reinterpret_cast<const float4*>(o_lat + ((size_t)rb * NH + h) * DC);
#pragma unroll
      for (int q = 0; q < 4; ++q) x[i][q] = ld_nc_v4(src + lane + 32 * q);
    }
    if (b0 + 8 * warp + 7 >= B) {  // a tile past the batch's end: zero those rows
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (b0 + 8 * warp + i >= B) x[i][q] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 8 * warp + i, rl = NT + r;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int f = lane + 32 * q;  // float4 index: columns 4f .. 4f + 3
        const float4 v = x[i][q];
        const float xs[4] = {v.x, v.y, v.z, v.w};
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(xs[2 * e]), h1 = __float2bfloat16_rn(xs[2 * e + 1]);
          hi[e] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
          lo[e] = pack_bf16x2(xs[2 * e] - __bfloat162float(h0), xs[2 * e + 1] - __bfloat162float(h1));
        }
        // chunk f / 16, 16-byte unit (f % 16) / 2, 8-byte half f % 2
        const uint32_t chunk = AO_B + (f >> 4) * AO_N * 128, u = (f & 15) >> 1, half = (f & 1) * 8;
        *reinterpret_cast<uint2*>(smem + chunk + r * 128 + ((u ^ (r & 7)) << 4) + half) =
            make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2*>(smem + chunk + rl * 128 + ((u ^ (rl & 7)) << 4) + half) =
            make_uint2(lo[0], lo[1]);
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int c = 0; ok && c < 8; ++c) {
      ok = wait_bar(bar_tma + 8 * c, 0, dev_status);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_ss(tmem, sdesc_sw128(sb + AO_A + c * 16384 + k * 32, 16, 1024),
               sdesc_sw128(sb + AO_B + c * AO_N * 128 + k * 32, 16, 1024), IDESC_AO,
               (c > 0 || k > 0) ? 1u : 0u);
    }
    mma_commit(bar_mma);  // also drains on failure
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  const bool done = __all_sync(0xffffffffu, wait_bar(bar_mma, 0, dev_status));  // warp-uniform for tcgen05.ld
  if (ok && done) {
    tc_fence_after();
    uint32_t vh[32], vl[32];
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16), vh);
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + NT, vl);
    tmem_ld_wait();
    const int col = h * DV + 32 * warp + lane;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (b0 + j >= B) continue;
      const float y = __uint_as_float(vh[j]) + __uint_as_float(vl[j]);
      const size_t i = (size_t)(b0 + j) * NH * DV + col;
      if (out_f32) reinterpret_cast<float*>(o)[i] = y;
      else reinterpret_cast<__nv_bfloat16*>(o)[i] = __float2bfloat16_rn(y);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, AO_N);
  }
}

// ------------------------------------------------ combine + absorb_out
// The split-KV merge (mla_combine) fused into absorb_out: each CTA merges
// the partial results of its 32 batch rows for its head straight into the
// B tile, writes the merged o_lat row and lse for the rows the plan split
// (and zeros / -inf for rows with an invalid length, as mla_combine does),
// then runs the absorb_out product. Same smem layout and MMA as
// absorb_out_kernel; 8 warps, each merging 4 rows, two rows at a time with
// all their loads in flight. The merge is mla_combine's arithmetic in the
// same order (bitwise the same o_lat and lse).
constexpr int AM_THREADS = 256;

__global__ void __launch_bounds__(AM_THREADS, 1)
    absorb_out_merge_kernel(const __grid_constant__ CUtensorMap tm_w, const char* __restrict__ ws,
                            WorkspaceLayout L, float* __restrict__ o_lat, float* __restrict__ lse,
                            void* __restrict__ o, int out_f32, int B, int32_t* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_tma = sb + AO_BAR, bar_mma = bar_tma + 8 * 8;  // 8 chunk barriers, then MMA
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + AO_BAR + 80);
  const int h = blockIdx.x, b0 = blockIdx.y * NT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqPlan* seqs = reinterpret_cast<const SeqPlan*>(ws + L.seqs);
  const float* lp = reinterpret_cast<const float*>(ws + L.lse_part);
  const float* op = reinterpret_cast<const float*>(ws + L.o_part);
  const bool p16 = reinterpret_cast<const PlanHeader*>(ws + L.header)->part_bf16 != 0;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    for (int c = 0; c < 9; ++c) mbar_init(bar_tma + 8 * c, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), AO_N);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (threadIdx.x == 0) {
    for (int c = 0; c < 8; ++c) {
      mbar_expect_tx(bar_tma + 8 * c, 16384);
      tma_load_2d(sb + AO_A + c * 16384, &tm_w, 64 * c, DV * h, bar_tma + 8 * c);
    }
  }

  constexpr int RS = 4;  // splits loaded per round
#pragma unroll 1
  for (int pr = 0; pr < 2; ++pr) {
    // rows ra, ra + 1 of the tile; a row past the batch reads row B - 1
    // and is dropped
    int n[2], sbeg[2], bb[2];
    bool valid[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = 4 * warp + 2 * pr + k;
      valid[k] = b0 + r < B;
      bb[k] = valid[k] ? b0 + r : B - 1;
      const SeqPlan sp = seqs[bb[k]];
      n[k] = valid[k] ? sp.n_splits : 0;
      sbeg[k] = sp.slot_begin;
    }
    // first batch of splits of both rows: a split past the end re-reads the last one
    // (weight 0); an unsplit row reads its o_lat row (weight 1)
    float4 x[2][RS][4];
    // float4 column lane + 32 q of split sidx of row k (partials in bf16 or
    // fp32 as the plan says), or of the row's o_lat if it was not split
    auto ld = [&](int k, int sidx, int q) -> float4 {
      const int c4 = lane + 32 * q;
      if (n[k] >= 2) {
        const size_t e0 = ((size_t)(sbeg[k] + min(sidx, n[k] - 1)) * NH + h) * DC;
        return p16 ? load_part_bf16x4(ws + L.o_part, e0 + 4 * (size_t)c4)
                   : ld_nc_v4(reinterpret_cast<const float4*>(op + e0) + c4);
      }
      return ld_nc_v4(reinterpret_cast<const float4*>(o_lat + ((size_t)bb[k] * NH + h) * DC) + c4);
    };
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int t = 0; t < RS; ++t)
#pragma unroll
        for (int q = 0; q < 4; ++q) x[k][t][q] = ld(k, t, q);
    float l_lane[2];
#pragma unroll
    for (int k = 0; k < 2; ++k)
      l_lane[k] = (n[k] >= 2 && lane < n[k]) ? lp[(size_t)(sbeg[k] + lane) * NH + h] : -INFINITY;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = 4 * warp + 2 * pr + k;
      float4 acc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      float m = -INFINITY, z = 0.f;
      if (n[k] == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = x[k][0][q];
      } else if (n[k] >= 2) {
        const int nk = n[k];
        m = l_lane[k];
        for (int s0 = 32; s0 < nk; s0 += 32)  // more than 32 splits: rare
          if (s0 + lane < nk) m = fmaxf(m, lp[(size_t)(sbeg[k] + s0 + lane) * NH + h]);
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o2));
        z = l_lane[k] == -INFINITY ? 0.f : expf(l_lane[k] - m);
        for (int s0 = 32; s0 < nk; s0 += 32)
          if (s0 + lane < nk) {
            const float l = lp[(size_t)(sbeg[k] + s0 + lane) * NH + h];
            z += l == -INFINITY ? 0.f : expf(l - m);
          }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o2);
        const float inv = 1.f / z;
        for (int s0 = 0; s0 < nk; s0 += RS) {
          if (s0 > 0) {  // later rounds (more than RS splits)
#pragma unroll
            for (int t = 0; t < RS; ++t)
#pragma unroll
              for (int q = 0; q < 4; ++q) x[k][t][q] = ld(k, s0 + t, q);
          }
#pragma unroll
          for (int t = 0; t < RS; ++t) {
            const int sidx = s0 + t;
            float l = __shfl_sync(0xffffffffu, l_lane[k], sidx & 31);
            if (sidx >= 32 && sidx < nk) l = lp[(size_t)(sbeg[k] + sidx) * NH + h];
            const float wgt = (sidx < nk && l != -INFINITY) ? expf(l - m) * inv : 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[q].x = fmaf(wgt, x[k][t][q].x, acc[q].x);
              acc[q].y = fmaf(wgt, x[k][t][q].y, acc[q].y);
              acc[q].z = fmaf(wgt, x[k][t][q].z, acc[q].z);
              acc[q].w = fmaf(wgt, x[k][t][q].w, acc[q].w);
            }
          }
        }
      }
      // merged (or invalid-length) rows: o_lat and lse as mla_combine writes them
      if (valid[k] && n[k] != 1) {
        float4* orow = reinterpret_cast<float4*>(o_lat + ((size_t)bb[k] * NH + h) * DC);
#pragma unroll
        for (int q = 0; q < 4; ++q) orow[lane + 32 * q] = acc[q];
        if (lane == 0) lse[(size_t)bb[k] * NH + h] = n[k] == 0 ? -INFINITY : m + logf(z);
      }
      // hi / lo split into the B tile (rows past the batch are zero)
      const int rl = NT + r;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = valid[k] ? acc[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float xs[4] = {v.x, v.y, v.z, v.w};
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(xs[2 * e]), h1 = __float2bfloat16_rn(xs[2 * e + 1]);
          hi[e] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
          lo[e] = pack_bf16x2(xs[2 * e] - __bfloat162float(h0), xs[2 * e + 1] - __bfloat162float(h1));
        }
        const int f = lane + 32 * q;
        const uint32_t chunk = AO_B + (f >> 4) * AO_N * 128, u = (f & 15) >> 1, half = (f & 1) * 8;
        *reinterpret_cast<uint2*>(smem + chunk + r * 128 + ((u ^ (r & 7)) << 4) + half) =
            make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2*>(smem + chunk + rl * 128 + ((u ^ (rl & 7)) << 4) + half) =
            make_uint2(lo[0], lo[1]);
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) {
#pragma unroll 1
    for (int c = 0; ok && c < 8; ++c) {
      ok = wait_bar(bar_tma + 8 * c, 0, dev_status);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_ss(tmem, sdesc_sw128(sb + AO_A + c * 16384 + k * 32, 16, 1024),
               sdesc_sw128(sb + AO_B + c * AO_N * 128 + k * 32, 16, 1024), IDESC_AO,
               (c > 0 || k > 0) ? 1u : 0u);
    }
    mma_commit(bar_mma);  // also drains on failure
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  const bool done = __all_sync(0xffffffffu, wait_bar(bar_mma, 0, dev_status));  // warp-uniform for tcgen05.ld
  if (warp < 4 && ok && done) {  // TMEM lanes 32 w .. 32 w + 31: warps 0-3
    tc_fence_after();
    uint32_t vh[32], vl[32];
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16), vh);
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + NT, vl);
    tmem_ld_wait();
    const int col = h * DV + 32 * warp + lane;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (b0 + j >= B) continue;
      const float y = __uint_as_float(vh[j]) + __uint_as_float(vl[j]);
      const size_t i = (size_t)(b0 + j) * NH * DV + col;
      if (out_f32) reinterpret_cast<float*>(o)[i] = y;
      else reinterpret_cast<__nv_bfloat16*>(o)[i] = __float2bfloat16_rn(y);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, AO_N);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 tensor map with 128-byte swizzle; dims/strides in elements/bytes.
cudaError_t make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return cudaErrorMisalignedAddress;
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult res = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tca

bool tc_absorb_supported(int n_h, int d_h, int d_r, int d_c, int d_v) {
  return n_h == tca::NH && d_h == tca::DH && d_r == tca::DR && d_c == tca::DC && d_v == tca::DV &&
         tc_decode_supported(n_h, d_c, d_r, 64);
}

cudaError_t tc_absorb_q_launch(const void* q, const void* w_uk, void* q_cat, int B,
                               int32_t* dev_status, cudaStream_t s) {
  CUtensorMap tm_w, tm_q;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)tca::DC, (cuuint64_t)tca::NH * tca::DH};
    const cuuint64_t strides[1] = {(cuuint64_t)tca::DC * 2};
    const cuuint32_t box[2] = {64, 128};
    cudaError_t e = tca::make_map(&tm_w, w_uk, 2, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)tca::QW, (cuuint64_t)tca::NH, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)tca::QW * 2, (cuuint64_t)tca::NH * tca::QW * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)tca::NT};
    cudaError_t e = tca::make_map(&tm_q, q, 3, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  static unsigned long long smem_done = 0;
  cudaError_t e = set_max_smem_once((const void*)tca::absorb_q_kernel, (int)tca::AQ_SMEM, smem_done);
  if (e != cudaSuccess) return e;
  const dim3 grid(tca::DC / 128, tca::NH, (B + tca::NT - 1) / tca::NT);
  tca::absorb_q_kernel<<<grid, 128, tca::AQ_SMEM, s>>>(
      tm_w, tm_q, reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<__nv_bfloat16*>(q_cat), B,
      dev_status);
  return cudaGetLastError();
}

cudaError_t tc_absorb_out_launch(const float* o_lat, const void* w_uv, void* o, int out_f32, int B,
                                 int32_t* dev_status, cudaStream_t s) {
  CUtensorMap tm_w;
  const cuuint64_t dims[2] = {(cuuint64_t)tca::DC, (cuuint64_t)tca::NH * tca::DV};
  const cuuint64_t strides[1] = {(cuuint64_t)tca::DC * 2};
  const cuuint32_t box[2] = {64, 128};
  cudaError_t e = tca::make_map(&tm_w, w_uv, 2, dims, strides, box);
  if (e != cudaSuccess) return e;
  static unsigned long long smem_done = 0;
  e = set_max_smem_once((const void*)tca::absorb_out_kernel, (int)tca::AO_SMEM, smem_done);
  if (e != cudaSuccess) return e;
  const dim3 grid(tca::NH, (B + tca::NT - 1) / tca::NT);
  tca::absorb_out_kernel<<<grid, 128, tca::AO_SMEM, s>>>(tm_w, o_lat, o, out_f32, B, dev_status);
  return cudaGetLastError();
}

cudaError_t tc_absorb_out_merge_launch(const void* ws, const WorkspaceLayout& L, float* o_lat,
                                       float* lse, const void* w_uv, void* o, int out_f32, int B,
                                       int32_t* dev_status, cudaStream_t s) {
  CUtensorMap tm_w;
  const cuuint64_t dims[2] = {(cuuint64_t)tca::DC, (cuuint64_t)tca::NH * tca::DV};
  const cuuint64_t strides[1] = {(cuuint64_t)tca::DC * 2};
  const cuuint32_t box[2] = {64, 128};
  cudaError_t e = tca::make_map(&tm_w, w_uv, 2, dims, strides, box);
  if (e != cudaSuccess) return e;
  static unsigned long long smem_done = 0;
  e = set_max_smem_once((const void*)tca::absorb_out_merge_kernel, (int)tca::AO_SMEM, smem_done);
  if (e != cudaSuccess) return e;
  const dim3 grid(tca::NH, (B + tca::NT - 1) / tca::NT);
  tca::absorb_out_merge_kernel<<<grid, tca::AM_THREADS, tca::AO_SMEM, s>>>(
      tm_w, reinterpret_cast<const char*>(ws), L, o_lat, lse, o, out_f32, B, dev_status);
  return cudaGetLastError();
}

}  // namespace mla
