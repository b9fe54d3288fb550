// tcgen05 decode attention over the paged latent cache, one CTA pair per
// worker, each page split between the two CTAs (DeepSeek-V2 shapes: 128
// heads, d_c = 512, d_R = 64, 64-token pages, bf16).
//
// Per page the 128 heads of a sequence share every cached row, so the work
// is two dense products on the 5th-generation tensor cores
// ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现", 3.2: the
// score is the latent-space content part plus the RoPE part; the latent
// output is the probability-weighted sum of cached latents):
//   S = Q_cat . Page^T      M = 128 heads, N = 64 tokens,  K = 576
//   O += P . Page[:, 0:512] M = 128 heads, N = 512 latent, K = 64 tokens
//
// The full O accumulator (128 x 512 fp32) would fill all of one SM's tensor
// memory, and the cache is read at HBM speed only when every SM streams
// bytes of its own, so each page is split between the two CTAs (SMs) of a
// cluster. CTA r of the pair loads, for every page:
//   latent columns [256 r, 256 r + 256) of all 64 tokens   (32 KB)
//   RoPE columns [512, 576) of tokens [32 r, 32 r + 32)     ( 4 KB)
// and computes from them a partial score matrix S_r (the latent part over
// its columns plus the RoPE part of its 32 tokens). The two CTAs swap S_r
// through distributed shared memory, both form S = S_0 + S_1 (the same fp32
// sum in both, so both take identical softmax decisions), and CTA r
// accumulates O[:, 256 r : 256 r + 256] = P . Page[:, its latent half] in
// its own tensor memory. No byte of the cache is loaded twice and no
// product is computed twice; only the softmax runs in both CTAs.
//
// Per CTA: 192 threads.
//   warp 0     TMA producer: latent half pages into a 5-stage ring, RoPE
//              quarter pages into a 4-slot ring; reads the block table.
//   warp 1     tcgen05 issuer (one thread), owns the TMEM allocation:
//              QK of page j+1 is issued before PV of page j.
//   warps 2-5  softmax: thread <-> head row <-> TMEM lane. Loads Q, swaps
//              S_r, computes P (bf16, into TMEM), rescales O, writes O / l.
// TMEM columns: O [0,256) fp32 | S [256,320) fp32 | Q latent half
// [320,448) bf16x2 | P [448,512) bf16x2, two buffers.
// SMEM: latent ring 160 KB | RoPE ring 16 KB | Q RoPE part 16 KB (A
// operand of the RoPE products) | received S 32 KB | barriers.
//
// Online softmax: running maximum in log2 units; O is rescaled only when a
// row's maximum grows by more than 8 (a factor 256). Until then P is taken
// against the stale maximum, which stays exact because l uses the same
// reference. Every mbarrier wait is bounded: after ~2 s it raises this CTA's
// abort flag and the peer's, reports MLA_DEV_TIMEOUT, and both CTAs drain
// their copies and MMAs and exit.
#include <cudaTypedefs.h>
#include <math.h>

#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_decode.h"

namespace mla {
namespace tcs {

using namespace ptx;

constexpr int NH = 128, DC = 512, DR = 64, ROW = DC + DR, PAGE = 64, HALF = DC / 2;
constexpr uint32_t CHUNK = PAGE * 128;   // 64 tokens x 64 columns (128 B rows)
constexpr uint32_t LSTAGE = 4 * CHUNK;   // latent half of a page
constexpr uint32_t RSLOT = 32 * 128;     // RoPE columns of 32 tokens
constexpr int NS = 5, NR = 4;            // ring depths
constexpr uint32_t QR_BYTES = NH * 128;  // Q RoPE part [128][64] bf16, swizzled
constexpr uint32_t XS_BYTES = NH * PAGE * 4;

constexpr uint32_t OFF_L = 0;
constexpr uint32_t OFF_R = OFF_L + NS * LSTAGE;
constexpr uint32_t OFF_QR = OFF_R + NR * RSLOT;
constexpr uint32_t OFF_XS = OFF_QR + QR_BYTES;
constexpr uint32_t OFF_BAR = OFF_XS + XS_BYTES;
enum {
  LFULL = 0,            // [NS] latent half page landed
  LEMPTY = NS,          // [NS] consumed by QK and PV
  RFULL = 2 * NS,       // [NR] RoPE quarter page landed
  REMPTY = RFULL + NR,  // [NR] consumed by QK
  QTMEM = REMPTY + NR,  // Q of the segment in TMEM and SMEM (4 warps)
  QEMPTY,               // last QK of a segment done
  SFULL,                // partial S in TMEM
  SFREE,                // partial S read by the 4 softmax warps
  XFULL,                // the peer's partial S landed here (armed here, bytes from the peer)
  XEMPTY,               // the peer read this CTA's partial S (4 remote warps)
  PFULL,                // [2] P buffer written (4 warps)
  ODONE = PFULL + 2,    // [2] PV from that P buffer done
  OFREE = ODONE + 2,    // O read out at a segment end (4 warps)
  FINAL,                // drain after an abort
  NBAR
};
constexpr uint32_t OFF_TSLOT = OFF_BAR + 8 * NBAR;
constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4;
static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
static_assert(OFF_R % 1024 == 0 && OFF_QR % 1024 == 0, "swizzled tiles need 1024-byte alignment");

constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 320, TM_P = 448, TM_COLS = 512;

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_QR = idesc_bf16_f32(128, 32, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, HALF, false, true);
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_NS = 100000000ull;

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
  int s, p0, p1, len, slot;
};

__device__ __forceinline__ bool seg_at(const WorkerPlan& w, const SeqPlan* seqs, int g, int s,
                                       Seg& out) {
  const SeqPlan sp = seqs[s];
  if (sp.pages == 0) return false;
  const int p0 = s == w.seq_begin ? w.page_begin : 0;
  const int p1 = s == w.seq_end ? w.page_end + 1 : sp.pages;
  if (p0 >= p1) return false;
  out.s = s;
  out.p0 = p0;
  out.p1 = p1;
  out.len = sp.len;
  out.slot = sp.n_splits > 1 ? sp.slot_begin + (g - sp.first_worker) : -1;
  return true;
}

struct Ctx {
  uint32_t bar0;
  volatile int* abort;
  uint32_t peer_abort;  // cluster address of the peer's abort flag
  int32_t* dev_status;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
  // Bounded waits; on failure also raise the peer's abort flag.
  __device__ bool wait(int i, uint32_t parity) const {
    if (mbar_wait_bounded(bar(i), parity, abort, dev_status, WAIT_NS)) return true;
    st_cluster_u32(peer_abort, 1);
    return false;
  }
  __device__ bool wait_cluster(int i, uint32_t parity) const {
    if (mbar_wait_cluster_bounded(bar(i), parity, abort, dev_status, WAIT_NS)) return true;
    st_cluster_u32(peer_abort, 1);
    return false;
  }
};

// Producer warp: for every page of the worker's range, in order, call
// `issue(k, block)` on lane 0 (k = page count so far), and `on_seq(s)` on
// lane 0 when sequence s starts. Lane-parallel block table reads; an
// out-of-range block id is reported and replaced by page 0.
template <typename F, typename G>
__device__ __forceinline__ bool for_each_page(const Params& p, const WorkerPlan& w,
                                              const SeqPlan* seqs, int g, int lane, F&& issue,
                                              G&& on_seq) {
  bool ok = true;
  uint32_t k = 0;
  for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
    Seg sg;
    if (!seg_at(w, seqs, g, s, sg)) continue;
    if (lane == 0) on_seq(s);
    for (int pb = sg.p0; ok && pb < sg.p1; pb += 32) {
      int blk = 0;
      if (pb + lane < sg.p1) {
        blk = p.block_table[(size_t)s * p.max_pages + pb + lane];
        if (blk < 0 || blk >= p.num_pages) {
          report(p.dev_status, MLA_DEV_BAD_BLOCK);
          blk = 0;
        }
      }
      const int n = min(32, sg.p1 - pb);
      for (int j = 0; ok && j < n; ++j, ++k) {
        const int bk = __shfl_sync(0xffffffffu, blk, j);
        if (lane == 0) ok = issue(k, bk);
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
  }
  return ok;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    tc_split_decode_kernel(const __grid_constant__ CUtensorMap tm_lat,
                           const __grid_constant__ CUtensorMap tm_rope, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t rank = cluster_ctarank();  // which half of every page
  const uint32_t peer = rank ^ 1u;
  const uint32_t sbase = smem_u32(smem);
  Ctx cx;
  cx.bar0 = sbase + OFF_BAR;
  cx.abort = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  cx.peer_abort = mapa_shared(sbase + OFF_ABORT, peer);
  cx.dev_status = p.dev_status;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x >> 1;
  const WorkerPlan w = reinterpret_cast<const WorkerPlan*>(p.ws + p.L.workers)[g];
  const SeqPlan* seqs = reinterpret_cast<const SeqPlan*>(p.ws + p.L.seqs);
  // Swizzled operand tiles need 1024-byte alignment of the shared window.
  const bool aligned = (sbase & 1023u) == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(cx.bar(LFULL + i), 1);
      mbar_init(cx.bar(LEMPTY + i), 1);
    }
    for (int i = 0; i < NR; ++i) {
      mbar_init(cx.bar(RFULL + i), 1);
      mbar_init(cx.bar(REMPTY + i), 1);
    }
    mbar_init(cx.bar(QTMEM), 4);
    mbar_init(cx.bar(QEMPTY), 1);
    mbar_init(cx.bar(SFULL), 1);
    mbar_init(cx.bar(SFREE), 4);
    mbar_init(cx.bar(XFULL), 1);
    mbar_expect_tx(cx.bar(XFULL), XS_BYTES);  // armed for the first page
    mbar_init(cx.bar(XEMPTY), 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(PFULL + i), 4);
      mbar_init(cx.bar(ODONE + i), 1);
    }
    mbar_init(cx.bar(OFREE), 4);
    mbar_init(cx.bar(FINAL), 1);
    *cx.abort = 0;
    if (!aligned) report(p.dev_status, MLA_DEV_TIMEOUT);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  cluster_sync_all();  // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (aligned && w.n_pages > 0) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_lat);
        tma_prefetch_desc(&tm_rope);
      }
      uint32_t issued = 0;
      const bool ok = for_each_page(
          p, w, seqs, g, lane,
          [&](uint32_t k, int bk) -> bool {
            const uint32_t st = k % NS, rs = k % NR;
            if (!cx.wait(LEMPTY + st, ((k / NS) & 1) ^ 1)) return false;
            mbar_expect_tx(cx.bar(LFULL + st), LSTAGE);
            for (int c = 0; c < 4; ++c)
              tma_load_2d(sbase + OFF_L + st * LSTAGE + c * CHUNK, &tm_lat,
                          (int)(HALF * rank) + 64 * c, bk * PAGE, cx.bar(LFULL + st));
            issued = 2 * k + 1;
            if (!cx.wait(REMPTY + rs, ((k / NR) & 1) ^ 1)) return false;
            mbar_expect_tx(cx.bar(RFULL + rs), RSLOT);
            tma_load_2d(sbase + OFF_R + rs * RSLOT, &tm_rope, DC, bk * PAGE + 32 * (int)rank,
                        cx.bar(RFULL + rs));
            issued = 2 * k + 2;
            return true;
          },
          [&](int s) {  // the next sequence's Q rows into L2 for their loads
            if (rank == 0 && s < w.seq_end)
              prefetch_l2(p.q_cat + (size_t)(s + 1) * NH * ROW, NH * ROW * 2);
          });
      if (!ok && lane == 0) {  // let issued copies land before the CTA exits
        const uint32_t pages = (issued + 1) / 2;
        for (uint32_t k = pages > (uint32_t)NS ? pages - NS : 0; k < pages; ++k)
          mbar_wait_drain(cx.bar(LFULL + k % NS), (k / NS) & 1, DRAIN_NS);
        const uint32_t rpages = issued / 2;
        for (uint32_t k = rpages > (uint32_t)NR ? rpages - NR : 0; k < rpages; ++k)
          mbar_wait_drain(cx.bar(RFULL + k % NR), (k / NR) & 1, DRAIN_NS);
      }
    } else if (warp == 1) {
      // ----------------------------------------------------------- MMA issue
      if (lane == 0) {
        uint32_t it = 0, seg = 0;
        bool ok = true;
        // PV of one page, from P buffer q & 1 and latent stage q % NS
        auto issue_pv = [&](uint32_t q, bool first, uint32_t qseg) -> bool {
          if (!cx.wait(PFULL + (q & 1), (q >> 1) & 1)) return false;
          if (first && qseg > 0 && !cx.wait(OFREE, (qseg - 1) & 1)) return false;
          tc_fence_after();
          const uint32_t vb = sbase + OFF_L + (q % NS) * LSTAGE;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + TM_O, tmem + TM_P + (q & 1) * 32 + kk * 8,
                   sdesc_sw128(vb + kk * 2048, CHUNK, 1024), IDESC_PV,
                   (first && kk == 0) ? 0u : 1u);
          mma_commit(cx.bar(LEMPTY + q % NS));
          mma_commit(cx.bar(ODONE + (q & 1)));
          return true;
        };
        bool have_pend = false, pend_first = false;
        uint32_t pend = 0, pend_seg = 0;
        for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
          Seg sg;
          if (!seg_at(w, seqs, g, s, sg)) continue;
          const int n = sg.p1 - sg.p0;
          ok = cx.wait(QTMEM, seg & 1);
          for (int j = 0; ok && j < n; ++j, ++it) {
            ok = cx.wait(SFREE, (it & 1) ^ 1) && cx.wait(LFULL + it % NS, (it / NS) & 1) &&
                 cx.wait(RFULL + it % NR, (it / NR) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t lb = sbase + OFF_L + (it % NS) * LSTAGE;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_ts(tmem + TM_S, tmem + TM_Q + kk * 8,
                     sdesc_sw128(lb + (kk >> 2) * CHUNK + (kk & 3) * 32, 16, 1024), IDESC_QK,
                     kk > 0 ? 1u : 0u);
            const uint32_t rb = sbase + OFF_R + (it % NR) * RSLOT;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + TM_S + 32 * rank, sdesc_sw128(sbase + OFF_QR + kk * 32, 16, 1024),
                     sdesc_sw128(rb + kk * 32, 16, 1024), IDESC_QR, 1u);
            mma_commit(cx.bar(REMPTY + it % NR));
            mma_commit(cx.bar(SFULL));
            if (j == n - 1) mma_commit(cx.bar(QEMPTY));
            if (have_pend) {
              ok = issue_pv(pend, pend_first, pend_seg);
              if (!ok) break;
            }
            have_pend = true;
            pend = it;
            pend_first = j == 0;
            pend_seg = seg;
          }
          ++seg;
        }
        if (ok && have_pend) ok = issue_pv(pend, pend_first, pend_seg);
        if (!ok) {  // every MMA issued so far completes before TMEM is freed
          mma_commit(cx.bar(FINAL));
          mbar_wait_drain(cx.bar(FINAL), 0, DRAIN_NS);
        }
      }
    } else {
      // ------------------------------------------------------------- softmax
      const int q4 = warp & 3;
      const int row = q4 * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      const uint32_t peer_xs = mapa_shared(sbase + OFF_XS, peer);
      const uint32_t peer_xfull = mapa_shared(cx.bar(XFULL), peer);
      const uint32_t peer_xempty = mapa_shared(cx.bar(XEMPTY), peer);
      const uint8_t* xs_own = smem + OFF_XS;
      float* o_part = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.o_part);
      float* lse_part = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.lse_part);
      const float c = p.scale_log2;
      // Q of sequence `qs`: latent half into TMEM, RoPE part into SMEM
      auto load_q = [&](int qs) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_cat + ((size_t)qs * NH + row) * ROW);
        uint4 qr[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) qr[u] = __ldg(src + DC / 8 + u);
#pragma unroll 1
        for (int c0 = 0; c0 < 4; c0 += 2) {
          uint4 x[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) x[u] = __ldg(src + (HALF * rank) / 8 + c0 * 8 + u);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              v[4 * u] = x[8 * h + u].x;
              v[4 * u + 1] = x[8 * h + u].y;
              v[4 * u + 2] = x[8 * h + u].z;
              v[4 * u + 3] = x[8 * h + u].w;
            }
            tmem_st32(lane_base + TM_Q + (c0 + h) * 32, v);
          }
        }
        uint8_t* qrow = smem + OFF_QR + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(qrow + ((u ^ (row & 7)) << 4)) = qr[u];
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(QTMEM));
      };
      // first sequence of the worker's range that owns pages at or after s0
      auto next_seg = [&](int s0, Seg& out) -> bool {
        for (int s = s0; s <= w.seq_end; ++s)
          if (seg_at(w, seqs, g, s, out)) return true;
        return false;
      };
      uint32_t it = 0, seg = 0;
      bool ok = true;
      Seg sg;
      bool have = next_seg(w.seq_begin, sg);
      if (have) load_q(sg.s);
      for (; ok && have; ++seg) {
        float m = -INFINITY, l = 0.f;
        const int n = sg.p1 - sg.p0;
        for (int j = 0; j < n; ++j, ++it) {
          // -- own partial S
          ok = __all_sync(0xffffffffu, cx.wait(SFULL, it & 1));
          if (!ok) break;
          tc_fence_after();
          uint32_t sa[32], sc[32];
          tmem_ld32(lane_base + TM_S, sa);
          tmem_ld32(lane_base + TM_S + 32, sc);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(cx.bar(SFREE));
          // -- swap partial S with the peer
          ok = __all_sync(0xffffffffu, cx.wait_cluster(XEMPTY, (it & 1) ^ 1));
          if (!ok) break;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            st_async_v4(peer_xs + (uint32_t)(i * NH + row) * 16, sa[4 * i], sa[4 * i + 1],
                        sa[4 * i + 2], sa[4 * i + 3], peer_xfull);
            st_async_v4(peer_xs + (uint32_t)((8 + i) * NH + row) * 16, sc[4 * i], sc[4 * i + 1],
                        sc[4 * i + 2], sc[4 * i + 3], peer_xfull);
          }
          ok = __all_sync(0xffffffffu, cx.wait_cluster(XFULL, it & 1));
          if (!ok) break;
          float sv[64];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(xs_own + (i * NH + row) * 16);
            const uint32_t* mine = i < 8 ? &sa[4 * i] : &sc[4 * (i - 8)];
            sv[4 * i] = __uint_as_float(mine[0]) + __uint_as_float(v.x);
            sv[4 * i + 1] = __uint_as_float(mine[1]) + __uint_as_float(v.y);
            sv[4 * i + 2] = __uint_as_float(mine[2]) + __uint_as_float(v.z);
            sv[4 * i + 3] = __uint_as_float(mine[3]) + __uint_as_float(v.w);
          }
          __syncwarp();
          if (lane == 0) {  // arm for the next page, then let the peer write it
            if (q4 == 0) mbar_expect_tx(cx.bar(XFULL), XS_BYTES);
            mbar_arrive_remote(peer_xempty);
          }

          // -- online softmax of the page
          const int nvalid = min(PAGE, sg.len - (sg.p0 + j) * PAGE);
          if (nvalid < PAGE) {  // ragged tail: -inf scores give p = 0
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i >= nvalid) sv[i] = -INFINITY;
          }
          float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
          for (int i = 4; i < 64; i += 4) {
            mx[0] = fmaxf(mx[0], sv[i]);
            mx[1] = fmaxf(mx[1], sv[i + 1]);
            mx[2] = fmaxf(mx[2], sv[i + 2]);
            mx[3] = fmaxf(mx[3], sv[i + 3]);
          }
          const float mp = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c;
          float m_use = m, alpha = 1.f;
          bool resc = false;
          if (j == 0) {
            m_use = mp;
          } else if (mp > m + 8.f) {
            m_use = mp;
            alpha = ex2_approx(m - mp);
            resc = true;
          }
          const float nm = -m_use;
          float sm[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float e0 = ex2_approx(fmaf(sv[2 * i], c, nm));
            const float e1 = ex2_approx(fmaf(sv[2 * i + 1], c, nm));
            sm[(2 * i) & 3] += e0;
            sm[(2 * i + 1) & 3] += e1;
            pk[i] = pack_bf16x2(e0, e1);
          }
          const float sum = (sm[0] + sm[1]) + (sm[2] + sm[3]);
          l = (j == 0) ? sum : fmaf(l, alpha, sum);
          m = m_use;

          // -- P buffer it & 1 is free once PV of page it - 2 is done
          ok = __all_sync(0xffffffffu, cx.wait(ODONE + (it & 1), ((it >> 1) & 1) ^ 1));
          if (!ok) break;
          if (__any_sync(0xffffffffu, resc)) {  // O *= alpha after PV of page it - 1
            ok = __all_sync(0xffffffffu, cx.wait(ODONE + ((it - 1) & 1), ((it - 1) >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < HALF / 32; ++cc) {
              uint32_t v[32];
              tmem_ld32(lane_base + TM_O + cc * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tmem_st32(lane_base + TM_O + cc * 32, v);
            }
          }
          tc_fence_after();
          tmem_st32(lane_base + TM_P + (it & 1) * 32, pk);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(cx.bar(PFULL + (it & 1)));
        }
        if (!ok) break;
        // -- the next sequence's Q, once the last QK of this one is done (the
        // QK of its first page then overlaps this epilogue)
        Seg nx;
        const bool have_next = next_seg(sg.s + 1, nx);
        if (have_next) {
          ok = __all_sync(0xffffffffu, cx.wait(QEMPTY, seg & 1));
          if (!ok) break;
          tc_fence_after();
          load_q(nx.s);
        }
        // -- epilogue: O / l for this CTA's latent half
        ok = __all_sync(0xffffffffu, cx.wait(ODONE + ((it - 1) & 1), ((it - 1) >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const float inv = 1.f / l;
        float* dst = (sg.slot < 0 ? p.o_lat + ((size_t)sg.s * NH + row) * DC
                                  : o_part + ((size_t)sg.slot * NH + row) * DC) +
                     HALF * rank;
#pragma unroll 1
        for (int cc = 0; cc < HALF / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(lane_base + TM_O + cc * 32, v);
          tmem_ld_wait();
          float4* d4 = reinterpret_cast<float4*>(dst + cc * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            d4[u] = make_float4(__uint_as_float(v[4 * u]) * inv, __uint_as_float(v[4 * u + 1]) * inv,
                                __uint_as_float(v[4 * u + 2]) * inv,
                                __uint_as_float(v[4 * u + 3]) * inv);
        }
        if (rank == 0) {
          const float lse = (m + log2f(l)) * 0.69314718055994531f;
          if (sg.slot < 0) p.lse[(size_t)sg.s * NH + row] = lse;
          else lse_part[(size_t)sg.slot * NH + row] = lse;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(OFREE));
        sg = nx;
        have = have_next;
      }
    }
  }
  __syncthreads();
  if (*cx.abort) {
    // stores this CTA sent to the peer complete on the peer's barrier; give
    // any still in flight time to land before the cluster may exit
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  cluster_sync_all();  // neither CTA leaves while the peer may still write into it
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// The paged cache [num_pages * 64][576] bf16 as 2-D tiles of `box_rows`
// rows x 64 columns with 128-byte swizzle.
cudaError_t make_cache_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return cudaErrorMisalignedAddress;
  const cuuint64_t dims[2] = {(cuuint64_t)ROW, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ROW * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult res = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Clusters of two that can be resident at once on the current device with
// this kernel's shared memory (0 if the query fails). Cached per device.
int max_clusters() {
  static int cached[64];
  static bool have[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (have[dev]) return cached[dev];
  if (cudaFuncSetAttribute(tc_split_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM_BYTES) != cudaSuccess)
    return 0;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2 > 0 ? sms / 2 : 1));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  int n = 0;
  // The kernel's cluster shape is fixed at compile time; some runtimes also
  // want it in the launch configuration.
  if (cudaOccupancyMaxActiveClusters(&n, tc_split_decode_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, tc_split_decode_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
  }
  cached[dev] = n;
  have[dev] = true;
  return n;
}

}  // namespace tcs

int tc_split_workers(int sms) {
  int n = sms / 2 > 0 ? sms / 2 : 1;
  const int mc = tcs::max_clusters();
  if (mc > 0 && mc < n) n = mc;
  return n;
}

cudaError_t tc_split_launch(const void* q_cat, const void* cache, const int32_t* block_table,
                            int max_pages, int num_pages, int workers, float scale, const void* ws,
                            const WorkspaceLayout& L, float* o_lat, float* lse,
                            int32_t* dev_status, cudaStream_t s) {
  CUtensorMap tm_lat, tm_rope;
  const uint64_t rows = (uint64_t)num_pages * tcs::PAGE;
  cudaError_t e = tcs::make_cache_map(&tm_lat, cache, rows, tcs::PAGE);
  if (e != cudaSuccess) return e;
  e = tcs::make_cache_map(&tm_rope, cache, rows, 32);
  if (e != cudaSuccess) return e;
  tcs::Params p;
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
  e = cudaFuncSetAttribute(tcs::tc_split_decode_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcs::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  tcs::tc_split_decode_kernel<<<2 * workers, 192, tcs::SMEM_BYTES, s>>>(tm_lat, tm_rope, p);
  return cudaGetLastError();
}

}  // namespace mla
