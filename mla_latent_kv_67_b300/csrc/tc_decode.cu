// tcgen05 decode attention over the paged latent cache (DeepSeek-V2 shapes:
// 128 heads, d_c = 512, d_R = 64, 64-token pages, bf16).
//
// The 128 heads of one sequence share every cached row, so per page the
// work is two dense products on the 5th-generation tensor cores:
//   S = Q_cat . Page^T     M = 128 heads, N = 64 tokens, K = 576
//   O += P . Page[:, lat]  M = 128 heads, N = 256 latent cols, K = 64 tokens
// ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现", 3.2: the
// score is the content part in the latent space plus the RoPE part; the
// latent output is the probability-weighted sum of cached latents.)
//
// Work split. A worker owns a contiguous range of the batch's pages (the
// plan). Each worker runs on two CTAs, one per SM: both compute the full S
// and the same softmax, and CTA r accumulates latent columns
// [256 r, 256 r + 256) of O. The whole O (128 x 512 fp32) would fill all of
// tensor memory and leave no room for S; half of it plus S plus part of Q
// fits in the 512 columns.
//
// Per CTA: 192 threads.
//   warp 0     TMA producer: 3 chunks of Q per sequence, 9 chunks (72 KB) per
//              page into a 2-stage ring; reads the block table.
//   warp 1     tcgen05 issuer (one thread); owns the TMEM allocation.
//   warps 2-5  softmax: thread <-> head row <-> TMEM lane. Each thread holds
//              its row's 64 scores, so the online softmax needs no
//              cross-thread reduction. Also writes Q's TMEM part, P (bf16,
//              swizzled) and the epilogue.
// TMEM columns: O [0,256) fp32 | S [256,320) fp32 | Q[:, 0:384] [320,512) bf16x2.
// SMEM: Q[:, 384:576] 48 KB | 2 page stages 144 KB | P 16 KB | barriers.
//
// Online softmax keeps a running max in log2 units and rescales O only when
// the max grows by more than 8 (a factor 256); until then probabilities are
// taken against the stale max, which stays exact because l uses the same
// reference. Every mbarrier wait is bounded: after ~2 s it raises an abort
// flag, reports MLA_DEV_TIMEOUT and the kernel drains and exits.
#include <cudaTypedefs.h>
#include <math.h>

#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_decode.h"

namespace mla {
namespace tcd {

using namespace ptx;

constexpr int NH = 128, DC = 512, DR = 64, ROW = DC + DR, PAGE = 64;
constexpr int NCHUNK = ROW / 64;           // 64-column (128-byte) chunks per row: 9
constexpr int QT_CHUNKS = 6;               // q_cat chunks 0..5 live in TMEM
constexpr int QS_CHUNKS = NCHUNK - QT_CHUNKS;
constexpr int HALF = DC / 2;
constexpr int STAGES = 2;

constexpr uint32_t PAGE_CHUNK_BYTES = PAGE * 128;              // 8 KB
constexpr uint32_t STAGE_BYTES = NCHUNK * PAGE_CHUNK_BYTES;    // 72 KB
constexpr uint32_t Q_CHUNK_BYTES = NH * 128;                   // 16 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_STAGE = OFF_Q + QS_CHUNKS * Q_CHUNK_BYTES;
constexpr uint32_t OFF_P = OFF_STAGE + STAGES * STAGE_BYTES;
constexpr uint32_t OFF_BAR = OFF_P + NH * 128;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;

constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 320, TM_COLS = 512;

enum {
  BAR_FULL = 0,        // [2] page stage loaded
  BAR_EMPTY = 2,       // [2] page stage consumed (QK and PV done)
  BAR_QFULL = 4,       // Q smem chunks loaded
  BAR_QTMEM = 5,       // Q tmem part written (4 warps)
  BAR_QEMPTY = 6,      // last QK of a sequence done: Q may be replaced
  BAR_SFULL = 7,       // S in TMEM
  BAR_SFREE = 8,       // S read by the softmax warps (4)
  BAR_PFULL = 9,       // P in SMEM and O corrected (4)
  BAR_ODONE = 10,      // PV of a page done
  BAR_OFREE = 11,      // epilogue read O (4)
  BAR_FINAL = 12,      // drain on abort
  NBAR = 13
};

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, HALF, false, true);
constexpr uint64_t WAIT_NS = 2000000000ull;

struct Params {
  const __nv_bfloat16* q_cat;
  const int32_t* block_table;
  const char* ws;
  WorkspaceLayout L;
  float* o_lat;
  float* lse;
  int32_t* dev_status;
  int max_pages, num_pages;
  float scale_log2;
};

// A sequence's share of a worker's page range.
struct Seg {
  int s, p0, p1, len, n_splits, slot;
};

__device__ __forceinline__ bool seg_at(const WorkerPlan& w, const SeqPlan* seqs, int g, int s, Seg& out) {
  const SeqPlan sp = seqs[s];
  if (sp.pages == 0) return false;
  const int p0 = s == w.seq_begin ? w.page_begin : 0;
  const int p1 = s == w.seq_end ? w.page_end + 1 : sp.pages;
  if (p0 >= p1) return false;
  out.s = s; out.p0 = p0; out.p1 = p1; out.len = sp.len; out.n_splits = sp.n_splits;
  out.slot = sp.n_splits > 1 ? sp.slot_begin + (g - sp.first_worker) : -1;
  return true;
}

__global__ void __launch_bounds__(192, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tm_cache,
                     const __grid_constant__ CUtensorMap tm_q, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * NBAR + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x >> 1;        // worker
  const int r = blockIdx.x & 1;         // latent half
  const WorkerPlan w = reinterpret_cast<const WorkerPlan*>(p.ws + p.L.workers)[g];
  const SeqPlan* seqs = reinterpret_cast<const SeqPlan*>(p.ws + p.L.seqs);

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_FULL), 1);
    mbar_init(bar(BAR_FULL + 1), 1);
    mbar_init(bar(BAR_EMPTY), 1);
    mbar_init(bar(BAR_EMPTY + 1), 1);
    mbar_init(bar(BAR_QFULL), 1);
    mbar_init(bar(BAR_QTMEM), 4);
    mbar_init(bar(BAR_QEMPTY), 1);
    mbar_init(bar(BAR_SFULL), 1);
    mbar_init(bar(BAR_SFREE), 4);
    mbar_init(bar(BAR_PFULL), 4);
    mbar_init(bar(BAR_ODONE), 1);
    mbar_init(bar(BAR_OFREE), 4);
    mbar_init(bar(BAR_FINAL), 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (w.n_pages > 0) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_cache);
        tma_prefetch_desc(&tm_q);
      }
      uint32_t it = 0, seg = 0;
      bool ok = true;
      for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
        Seg sg;
        if (!seg_at(w, seqs, g, s, sg)) continue;
        if (lane == 0) {
          ok = mbar_wait_bounded(bar(BAR_QEMPTY), (seg & 1) ^ 1, abort_flag, p.dev_status, WAIT_NS);
          if (ok) {
            mbar_expect_tx(bar(BAR_QFULL), QS_CHUNKS * Q_CHUNK_BYTES);
            for (int j = 0; j < QS_CHUNKS; ++j)
              tma_load_2d(sbase + OFF_Q + j * Q_CHUNK_BYTES, &tm_q, (QT_CHUNKS + j) * 64, s * NH,
                          bar(BAR_QFULL));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        for (int pb = sg.p0; ok && pb < sg.p1; pb += 32) {
          int blk = 0;
          if (pb + lane < sg.p1) {
            blk = p.block_table[(size_t)s * p.max_pages + pb + lane];
            if (blk < 0 || blk >= p.num_pages) {
              report(p.dev_status, MLA_DEV_BAD_BLOCK);
              blk = 0;  // read a valid page instead; the result is flagged
            }
          }
          const int n = min(32, sg.p1 - pb);
          for (int k = 0; ok && k < n; ++k, ++it) {
            const int bk = __shfl_sync(0xffffffffu, blk, k);
            if (lane == 0) {
              const uint32_t st = it & 1;
              ok = mbar_wait_bounded(bar(BAR_EMPTY + st), ((it >> 1) & 1) ^ 1, abort_flag,
                                     p.dev_status, WAIT_NS);
              if (ok) {
                const uint32_t dst = sbase + OFF_STAGE + st * STAGE_BYTES;
                mbar_expect_tx(bar(BAR_FULL + st), STAGE_BYTES);
                for (int c = 0; c < NCHUNK; ++c)
                  tma_load_2d(dst + c * PAGE_CHUNK_BYTES, &tm_cache, c * 64, bk * PAGE,
                              bar(BAR_FULL + st));
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
          }
        }
        ++seg;
      }
      // On abort, let the copies already issued land before the CTA exits.
      if (!ok && lane == 0) {
        for (uint32_t k = it > 2 ? it - 2 : 0; k < it; ++k)
          mbar_wait_bounded(bar(BAR_FULL + (k & 1)), (k >> 1) & 1, abort_flag, nullptr, WAIT_NS);
      }
    } else if (warp == 1) {
      // ----------------------------------------------------------- MMA issue
      if (lane == 0) {
        uint32_t it = 0, seg = 0;
        bool ok = true;
        auto issue_qk = [&](uint32_t i) -> bool {
          const uint32_t st = i & 1;
          if (!mbar_wait_bounded(bar(BAR_FULL + st), (i >> 1) & 1, abort_flag, p.dev_status, WAIT_NS))
            return false;
          if (!mbar_wait_bounded(bar(BAR_SFREE), (i & 1) ^ 1, abort_flag, p.dev_status, WAIT_NS))
            return false;
          tc_fence_after();
          const uint32_t pg = sbase + OFF_STAGE + st * STAGE_BYTES;
#pragma unroll 1
          for (int kk = 0; kk < 4 * QT_CHUNKS; ++kk) {
            const uint64_t bd = sdesc_sw128(pg + (kk >> 2) * PAGE_CHUNK_BYTES + (kk & 3) * 32, 16, 1024);
            mma_ts(tmem + TM_S, tmem + TM_Q + kk * 8, bd, IDESC_QK, kk > 0);
          }
#pragma unroll 1
          for (int kk = 4 * QT_CHUNKS; kk < 4 * NCHUNK; ++kk) {
            const int c = kk >> 2;
            const uint64_t ad = sdesc_sw128(sbase + OFF_Q + (c - QT_CHUNKS) * Q_CHUNK_BYTES + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(pg + c * PAGE_CHUNK_BYTES + (kk & 3) * 32, 16, 1024);
            mma_ss(tmem + TM_S, ad, bd, IDESC_QK, 1);
          }
          mma_commit(bar(BAR_SFULL));
          return true;
        };
        for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
          Seg sg;
          if (!seg_at(w, seqs, g, s, sg)) continue;
          ok = mbar_wait_bounded(bar(BAR_QFULL), seg & 1, abort_flag, p.dev_status, WAIT_NS) &&
               mbar_wait_bounded(bar(BAR_QTMEM), seg & 1, abort_flag, p.dev_status, WAIT_NS) &&
               (seg == 0 || mbar_wait_bounded(bar(BAR_OFREE), (seg - 1) & 1, abort_flag, p.dev_status, WAIT_NS));
          if (!ok) break;
          tc_fence_after();
          const int n = sg.p1 - sg.p0;
          ok = issue_qk(it);
          for (int j = 0; ok && j < n; ++j, ++it) {
            if (j + 1 < n) {
              ok = issue_qk(it + 1);
              if (!ok) break;
            } else {
              mma_commit(bar(BAR_QEMPTY));
            }
            ok = mbar_wait_bounded(bar(BAR_PFULL), it & 1, abort_flag, p.dev_status, WAIT_NS);
            if (!ok) break;
            tc_fence_after();
            const uint32_t st = it & 1;
            const uint32_t pg = sbase + OFF_STAGE + st * STAGE_BYTES + (4 * r) * PAGE_CHUNK_BYTES;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc_sw128(sbase + OFF_P + kk * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(pg + kk * 2048, PAGE_CHUNK_BYTES, 1024);
              mma_ss(tmem + TM_O, ad, bd, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar(BAR_EMPTY + st));
            mma_commit(bar(BAR_ODONE));
          }
          ++seg;
        }
        if (!ok) {  // drain: every MMA issued so far completes before TMEM is freed
          mma_commit(bar(BAR_FINAL));
          mbar_wait_bounded(bar(BAR_FINAL), 0, abort_flag, nullptr, WAIT_NS);
        }
      }
    } else {
      // ------------------------------------------------------------- softmax
      const int q4 = warp & 3;
      const int row = q4 * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      uint32_t it = 0, seg = 0;
      bool ok = true;
      float* o_part = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.o_part);
      float* lse_part = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.lse_part);
      for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
        Seg sg;
        if (!seg_at(w, seqs, g, s, sg)) continue;
        // Q[:, 0:384] of this sequence into TMEM (row = lane)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(BAR_QEMPTY), (seg & 1) ^ 1, abort_flag, p.dev_status, WAIT_NS));
        if (!ok) break;
        tc_fence_after();
        {
          const uint4* src = reinterpret_cast<const uint4*>(p.q_cat + ((size_t)s * NH + row) * ROW);
#pragma unroll 1
          for (int c = 0; c < QT_CHUNKS; ++c) {
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 x = __ldg(src + c * 8 + u);
              v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
            }
            tmem_st32(lane_base + TM_Q + c * 32, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_QTMEM));

        float m = -INFINITY, l = 0.f;
        const int n = sg.p1 - sg.p0;
        for (int j = 0; j < n; ++j, ++it) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(BAR_SFULL), it & 1, abort_flag, p.dev_status, WAIT_NS));
          if (!ok) break;
          tc_fence_after();
          uint32_t sa[32], sb[32];
          tmem_ld32(lane_base + TM_S, sa);
          tmem_ld32(lane_base + TM_S + 32, sb);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_SFREE));

          const int nvalid = min(PAGE, sg.len - (sg.p0 + j) * PAGE);
          float x[64];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = i < nvalid ? __uint_as_float(sa[i]) * p.scale_log2 : -INFINITY;
            x[32 + i] = 32 + i < nvalid ? __uint_as_float(sb[i]) * p.scale_log2 : -INFINITY;
          }
          float mp = x[0];
#pragma unroll
          for (int i = 1; i < 64; ++i) mp = fmaxf(mp, x[i]);
          float m_use = m, alpha = 1.f;
          bool rescale = false;
          if (j == 0) {
            m_use = mp;
          } else if (mp > m + 8.f) {
            m_use = mp;
            alpha = exp2f(m - mp);
            rescale = true;
          }
          float sum = 0.f;
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float e0 = exp2f(x[2 * i] - m_use), e1 = exp2f(x[2 * i + 1] - m_use);
            sum += e0 + e1;
            pk[i] = pack_bf16x2(e0, e1);
          }
          l = (j == 0) ? sum : l * alpha + sum;
          m = m_use;
          if (j > 0) {  // PV of the previous page done: P buffer free, O stable
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(BAR_ODONE), (it - 1) & 1, abort_flag, p.dev_status, WAIT_NS));
            if (!ok) break;
            tc_fence_after();
            if (rescale) {
#pragma unroll 1
              for (int c = 0; c < HALF / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(lane_base + TM_O + c * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                tmem_st32(lane_base + TM_O + c * 32, v);
              }
              tmem_st_wait();
            }
          }
          uint8_t* prow = smem + OFF_P + row * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(prow + ((u ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_PFULL));
        }
        if (!ok) break;
        // epilogue: O / l for this CTA's latent half
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(BAR_ODONE), (it - 1) & 1, abort_flag, p.dev_status, WAIT_NS));
        if (!ok) break;
        tc_fence_after();
        const float inv = 1.f / l;
        float* dst = sg.slot < 0 ? p.o_lat + ((size_t)sg.s * NH + row) * DC + r * HALF
                                 : o_part + ((size_t)sg.slot * NH + row) * DC + r * HALF;
#pragma unroll 1
        for (int c = 0; c < HALF / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + TM_O + c * 32, v);
          tmem_ld_wait();
          float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            d4[u] = make_float4(__uint_as_float(v[4 * u]) * inv, __uint_as_float(v[4 * u + 1]) * inv,
                                __uint_as_float(v[4 * u + 2]) * inv, __uint_as_float(v[4 * u + 3]) * inv);
        }
        if (r == 0) {
          const float lse = (m + log2f(l)) * 0.69314718055994531f;
          if (sg.slot < 0) p.lse[(size_t)sg.s * NH + row] = lse;
          else lse_part[(size_t)sg.slot * NH + row] = lse;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_OFREE));
        ++seg;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// One page, no softmax: S = Q . Page^T and O = P . Page[:, 256 r : 256 r + 256]
// with the same operand layouts, descriptors and instructions as the decode
// kernel. A diagnostic for the tensor-core data path.
__global__ void __launch_bounds__(192, 1)
    tc_selftest_kernel(const __grid_constant__ CUtensorMap tm_cache,
                       const __grid_constant__ CUtensorMap tm_q, const __nv_bfloat16* q_cat,
                       const __nv_bfloat16* pmat, float* s_out, float* o_out, int r,
                       int32_t* dev_status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * NBAR + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t b_tma = bar0, b_q = bar0 + 8, b_mma = bar0 + 16;
  if (threadIdx.x == 0) {
    mbar_init(b_tma, 1);
    mbar_init(b_q, 4);
    mbar_init(b_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(b_tma, QS_CHUNKS * Q_CHUNK_BYTES + STAGE_BYTES);
      for (int j = 0; j < QS_CHUNKS; ++j)
        tma_load_2d(sbase + OFF_Q + j * Q_CHUNK_BYTES, &tm_q, (QT_CHUNKS + j) * 64, 0, b_tma);
      for (int c = 0; c < NCHUNK; ++c)
        tma_load_2d(sbase + OFF_STAGE + c * PAGE_CHUNK_BYTES, &tm_cache, c * 64, 0, b_tma);
      mbar_wait_bounded(b_tma, 0, abort_flag, dev_status, WAIT_NS);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const bool ok = mbar_wait_bounded(b_tma, 0, abort_flag, dev_status, WAIT_NS) &&
                      mbar_wait_bounded(b_q, 0, abort_flag, dev_status, WAIT_NS);
      if (ok) {
        tc_fence_after();
        const uint32_t pg = sbase + OFF_STAGE;
        for (int kk = 0; kk < 4 * QT_CHUNKS; ++kk) {
          const uint64_t bd = sdesc_sw128(pg + (kk >> 2) * PAGE_CHUNK_BYTES + (kk & 3) * 32, 16, 1024);
          mma_ts(tmem + TM_S, tmem + TM_Q + kk * 8, bd, IDESC_QK, kk > 0);
        }
        for (int kk = 4 * QT_CHUNKS; kk < 4 * NCHUNK; ++kk) {
          const int c = kk >> 2;
          const uint64_t ad = sdesc_sw128(sbase + OFF_Q + (c - QT_CHUNKS) * Q_CHUNK_BYTES + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(pg + c * PAGE_CHUNK_BYTES + (kk & 3) * 32, 16, 1024);
          mma_ss(tmem + TM_S, ad, bd, IDESC_QK, 1);
        }
        const uint32_t pv = pg + (4 * r) * PAGE_CHUNK_BYTES;
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc_sw128(sbase + OFF_P + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(pv + kk * 2048, PAGE_CHUNK_BYTES, 1024);
          mma_ss(tmem + TM_O, ad, bd, IDESC_PV, kk > 0);
        }
      }
      mma_commit(b_mma);
    }
  } else {
    const int q4 = warp & 3, row = q4 * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint4* src = reinterpret_cast<const uint4*>(q_cat + (size_t)row * ROW);
    for (int c = 0; c < QT_CHUNKS; ++c) {
      uint32_t v[32];
      for (int u = 0; u < 8; ++u) {
        const uint4 x = src[c * 8 + u];
        v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
      }
      tmem_st32(lane_base + TM_Q + c * 32, v);
    }
    tmem_st_wait();
    const uint4* prow_src = reinterpret_cast<const uint4*>(pmat + (size_t)row * 64);
    uint8_t* prow = smem + OFF_P + row * 128;
    for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(prow + ((u ^ (row & 7)) << 4)) = prow_src[u];
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(b_q);
    if (mbar_wait_bounded(b_mma, 0, abort_flag, dev_status, WAIT_NS)) {
      tc_fence_after();
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_base + TM_S + c * 32, v);
        tmem_ld_wait();
        for (int i = 0; i < 32; ++i) s_out[row * 64 + c * 32 + i] = __uint_as_float(v[i]);
      }
      for (int c = 0; c < HALF / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_base + TM_O + c * 32, v);
        tmem_ld_wait();
        for (int i = 0; i < 32; ++i) o_out[row * HALF + c * 32 + i] = __uint_as_float(v[i]);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Row-major bf16 matrix [rows][576] seen as 2-D tiles of box_rows x 64
// columns with 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return cudaErrorMisalignedAddress;
  const cuuint64_t dims[2] = {(cuuint64_t)ROW, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ROW * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult res = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool device_is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

}  // namespace tcd

bool tc_decode_supported(int n_h, int d_c, int d_r, int page_size) {
  return n_h == tcd::NH && d_c == tcd::DC && d_r == tcd::DR && page_size == tcd::PAGE &&
         tcd::device_is_sm103();
}

int tc_decode_workers(int sms) { return sms / 2 > 0 ? sms / 2 : 1; }

cudaError_t tc_decode_launch(const void* q_cat, const void* cache, const int32_t* block_table,
                             int max_pages, int num_pages, int B, int workers, float scale,
                             const void* ws, const WorkspaceLayout& L, float* o_lat, float* lse,
                             int32_t* dev_status, cudaStream_t s) {
  CUtensorMap tm_cache, tm_q;
  cudaError_t e = tcd::make_map(&tm_cache, cache, (uint64_t)num_pages * tcd::PAGE, tcd::PAGE);
  if (e != cudaSuccess) return e;
  e = tcd::make_map(&tm_q, q_cat, (uint64_t)B * tcd::NH, tcd::NH);
  if (e != cudaSuccess) return e;
  tcd::Params p;
  p.q_cat = reinterpret_cast<const __nv_bfloat16*>(q_cat);
  p.block_table = block_table;
  p.ws = reinterpret_cast<const char*>(ws);
  p.L = L;
  p.o_lat = o_lat;
  p.lse = lse;
  p.dev_status = dev_status;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  e = cudaFuncSetAttribute(tcd::tc_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tcd::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  tcd::tc_decode_kernel<<<2 * workers, 192, tcd::SMEM_BYTES, s>>>(tm_cache, tm_q, p);
  return cudaGetLastError();
}

cudaError_t tc_selftest_launch(const void* q_cat, const void* page, const void* pmat, float* s_out,
                               float* o_out, int r, int32_t* dev_status, cudaStream_t s) {
  CUtensorMap tm_cache, tm_q;
  cudaError_t e = tcd::make_map(&tm_cache, page, tcd::PAGE, tcd::PAGE);
  if (e != cudaSuccess) return e;
  e = tcd::make_map(&tm_q, q_cat, tcd::NH, tcd::NH);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tcd::tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tcd::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  tcd::tc_selftest_kernel<<<1, 192, tcd::SMEM_BYTES, s>>>(
      tm_cache, tm_q, reinterpret_cast<const __nv_bfloat16*>(q_cat),
      reinterpret_cast<const __nv_bfloat16*>(pmat), s_out, o_out, r, dev_status);
  return cudaGetLastError();
}

}  // namespace mla
