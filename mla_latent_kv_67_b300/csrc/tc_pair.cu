// tcgen05 decode attention over the paged latent cache, one CTA pair per
// worker (DeepSeek-V2 shapes: 128 heads, d_c = 512, d_R = 64, 64-token
// pages, bf16).
//
// Per page the 128 heads of a sequence share every cached row, so the work
// is two dense products on the 5th-generation tensor cores
// ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现", 3.2: the
// score is the latent-space content part plus the RoPE part; the latent
// output is the probability-weighted sum of cached latents):
//   S = Q_cat . Page^T      M = 128 heads, N = 64 tokens,  K = 576
//   O += P . Page[:, 0:512] M = 128 heads, N = 512 latent, K = 64 tokens
// The full O accumulator (128 x 512 fp32) fills all 512 columns of one SM's
// tensor memory, so one SM cannot hold O together with Q and S. The two
// products therefore run on the two CTAs (two SMs) of a cluster, each once:
//
//   rank 0, the score CTA: Q_cat in TMEM as the A operand, S into TMEM
//     (two buffers), pages from a 3-stage ring; two MMA issuer threads
//     take pages in turn (page i into S buffer i % 2). One thread issues
//     N = 64 products at about half the tensor core's rate; two issuing
//     threads together nearly saturate it, and a third only lengthens every
//     page's product chain (and so how long it holds its ring stage). Two groups of four
//     softmax warps take the pages in turn (thread = head row = TMEM lane;
//     the groups share each page's reference maximum through shared
//     memory) and turn S into bf16 probabilities P and
//     store them, with per-row rescale factors, straight from registers into
//     the value CTA's shared memory (st.async, completion counted in bytes on
//     the value CTA's barrier). A sequence's Q_cat rows (128 x 576, the same
//     shape as two pages) travel through the same ring as two items ahead of
//     its pages, so the TMA engine fetches them and the softmax warps only
//     move them from shared memory into TMEM.
//   rank 1, the value CTA: O in TMEM (all 512 columns), the pages' latent
//     part from its own 2-stage ring, P from one of three slots. The MMA
//     issuer alone watches the P slots: it re-arms a slot's barrier, frees
//     the slot with a commit straight to the score CTA's barrier, and hands
//     the eight epilogue warps a command only when O needs work (a rescale,
//     or a finished sequence). The epilogue warps sleep otherwise: every
//     extra thread polling a barrier that 1,300 st.async completions per
//     page also update slows the whole SM down. At a sequence's end the two
//     groups of four write O / l, one 256-column half each, through a
//     swizzled shared-memory transpose, so every warp store covers whole
//     rows; each half is handed back to the next sequence's products as
//     soon as it is written out. (One SM stores only ~50 GB/s, so the 256 KB
//     of O take ~5 us however many warps write them.)
//
// Each CTA loads its pages on its own: the second read of a page hits L2 and
// costs no HBM bandwidth, and neither ring waits for the other. The MMA
// issuers synchronise once per page (one barrier wait, one fence, one commit
// per stage).
//
// Online softmax: running maximum in log2 units; O is rescaled only when a
// row's maximum grows by more than 8 (a factor 256). Until then P is taken
// against the stale maximum, which stays exact because l uses the same
// reference.
//
// Every mbarrier wait is bounded: after ~2 s it raises the CTA's abort flag
// and the peer's, reports MLA_DEV_TIMEOUT, and both CTAs drain their copies
// and MMAs and exit.
#include <cudaTypedefs.h>
#include <math.h>

#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_decode.h"

namespace mla {
namespace tcp {

using namespace ptx;

constexpr int NH = 128, DC = 512, DR = 64, ROW = DC + DR, PAGE = 64;
constexpr int NCHUNK = ROW / 64;  // 64-column (128-byte) chunks per cached row: 9
constexpr int VCHUNK = DC / 64;   // latent chunks: 8
constexpr uint32_t CHUNK = PAGE * 128;  // one chunk of a page: 64 tokens x 128 B
constexpr int NKS = 3;                  // score CTA: page stages
constexpr int NVS = 2;                  // value CTA: latent page stages
constexpr int NP = 3;                   // P slots
constexpr int NSB = 2;                  // S buffers in TMEM
constexpr int NQK = 2;                  // QK issuer threads (page i: issuer and S buffer i % 2)
static_assert(NQK == NSB, "each QK issuer owns one S buffer");
constexpr uint32_t KSTAGE = NCHUNK * CHUNK;
constexpr int HALF_BLOCKS = DC / 2 / 32;  // 32-column TMEM blocks in one half of O
constexpr uint32_t VSTAGE = VCHUNK * CHUNK;
// P [128][64] bf16 in the non-swizzled core-matrix layout: the 16-byte
// group u (tokens 8u..8u+7) of head row r sits at u * P_KGROUP + 16 r, so a
// warp's store of one group covers 512 contiguous bytes.
constexpr uint32_t P_BYTES = NH * 128;
constexpr uint32_t P_KGROUP = NH * 16;
// per P slot: alpha[128], inv_l[128] (float), one rescale flag per softmax warp
constexpr uint32_t XOFF_ALPHA = 0, XOFF_INVL = 4 * NH, XOFF_FLAG = 8 * NH;
constexpr uint32_t X_BYTES = XOFF_FLAG + 16;
constexpr uint32_t P_TX = P_BYTES + X_BYTES;  // bytes that fill one P slot

// score CTA shared memory
constexpr uint32_t S_OFF_K = 0;
// the two softmax groups' hand-over: the reference maximum each page used
// ([2][NH], by page parity), and at a sequence's end the l and reference of
// the group that does not own the last page ([2][NH] each)
constexpr uint32_t S_OFF_MREF = S_OFF_K + NKS * KSTAGE;
constexpr uint32_t S_OFF_LX = S_OFF_MREF + 2 * NH * 4;
constexpr uint32_t S_OFF_BAR = S_OFF_LX + 4 * NH * 4;
enum {
  KFULL = 0,             // [NKS] ring item (page or Q half) landed
  KEMPTY = NKS,          // [NKS] ring item consumed (4 arrivals)
  SFULL = 2 * NKS,       // [NSB] S buffer written
  SFREE = SFULL + NSB,   // [NSB] S buffer read by the 4 softmax warps
  QTMEM = SFREE + NSB,   // Q of the segment in TMEM (4 warps)
  QEMPTY = QTMEM + 1,    // last QK of a segment done
  PEMPTY = QEMPTY + 1,   // [NP] value CTA done with P slot (its PV commit)
  SFINAL = PEMPTY + NP,  // [NQK] drain after an abort (one per QK issuer)
  MREADY = SFINAL + NQK, // [2] reference maximum of a page published (4 warps), by page parity
  LXREADY = MREADY + 2,  // [2] l of the non-last group published at a sequence's end (4 warps)
  S_NBAR = LXREADY + 2
};
constexpr uint32_t S_OFF_TSLOT = S_OFF_BAR + 8 * S_NBAR;
constexpr uint32_t S_OFF_ABORT = S_OFF_TSLOT + 4;
constexpr uint32_t S_SMEM = S_OFF_ABORT + 4;

// value CTA shared memory
constexpr uint32_t V_OFF_V = 0;
constexpr uint32_t V_OFF_P = V_OFF_V + NVS * VSTAGE;   // NP P slots
constexpr uint32_t V_OFF_X = V_OFF_P + NP * P_BYTES;   // NP extras slots
constexpr uint32_t V_OFF_STG = V_OFF_X + NP * X_BYTES;  // 8 warps x 32 rows x 128 B
constexpr uint32_t V_OFF_XA = V_OFF_STG + 8 * 32 * 128;  // alpha of a rescale command
constexpr uint32_t V_OFF_XL = V_OFF_XA + 4 * NH;  // [2] 1 / l of a finished sequence (by its parity)
constexpr uint32_t V_OFF_CMD = V_OFF_XL + 8 * NH;  // command: kind, page index
constexpr uint32_t V_OFF_BAR = V_OFF_CMD + 16;
enum {
  VFULL = 0,            // [NVS] latent page landed
  VEMPTY = NVS,         // [NVS] latent page consumed by PV
  PFULL = 2 * NVS,      // [NP] P slot filled (armed here, bytes from the score CTA)
  ODONE = PFULL + NP,   // [NP] PV from that P slot done
  ORESC = ODONE + NP,   // O rescaled by epilogue group 0
  WORK = ORESC + 1,     // a command for epilogue group 0 (issuer)
  EPI = WORK + 1,       // sequence finished (group 0 to group 1)
  OFREE = EPI + 1,      // [2] a column half of O read out by its 4 warps
  VFINAL = OFREE + 2,   // drain after an abort
  V_NBAR = VFINAL + 1
};
constexpr uint32_t V_OFF_TSLOT = V_OFF_BAR + 8 * V_NBAR;
constexpr uint32_t V_OFF_ABORT = V_OFF_TSLOT + 4;
constexpr uint32_t V_SMEM = V_OFF_ABORT + 4;

constexpr uint32_t SMEM_BYTES = S_SMEM > V_SMEM ? S_SMEM : V_SMEM;
static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
static_assert(V_OFF_P % 1024 == 0 && X_BYTES % 16 == 0 && V_OFF_STG % 16 == 0 && V_OFF_BAR % 8 == 0,
              "layout alignment");

// TMEM columns. Score CTA: S0 | S1 | Q (576 bf16 packed in 288 columns).
constexpr uint32_t TM_S = 0, TM_Q = 64 * NSB, TM_COLS = 512;
static_assert(TM_Q + 288 <= TM_COLS, "score CTA TMEM budget");

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 256, false, true);
#ifdef MLA_TEST_HOOKS
constexpr uint64_t WAIT_NS = 20000000ull;  // test build: a withheld item times out in 20 ms
#else
constexpr uint64_t WAIT_NS = 2000000000ull;
#endif
constexpr uint64_t DRAIN_NS = 100000000ull;

struct Params {
  const int32_t* block_table;
  const char* ws;
  WorkspaceLayout L;
  float* o_lat;
  float* lse;
  int32_t* dev_status;
  int max_pages, num_pages;
  float scale_log2;
  int bt_div;  // new tokens per sequence: query row s uses block-table row s / bt_div
  int withhold;  // read by the test build only: the score CTA's producer issues nothing
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

// First sequence at or after s0 in the worker's range that owns pages.
__device__ __forceinline__ bool next_seg(const WorkerPlan& w, const SeqPlan* seqs, int g, int s0,
                                         Seg& out) {
  for (int s = s0; s <= w.seq_end; ++s)
    if (seg_at(w, seqs, g, s, out)) return true;
  return false;
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
  __device__ bool wait_sleepy(int i, uint32_t parity) const {
    if (mbar_wait_sleepy(bar(i), parity, abort, dev_status, WAIT_NS, 256)) return true;
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
// lane 0 when sequence s starts; either returning false stops the walk.
// Lane-parallel block table reads; an out-of-range block id is reported and
// replaced by page 0.
template <typename F, typename G>
__device__ __forceinline__ bool for_each_page(const Params& p, const WorkerPlan& w,
                                              const SeqPlan* seqs, int g, int lane, F&& issue,
                                              G&& on_seq) {
  bool ok = true;
  uint32_t k = 0;
  for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
    Seg sg;
    if (!seg_at(w, seqs, g, s, sg)) continue;
    if (lane == 0) ok = on_seq(s);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    for (int pb = sg.p0; ok && pb < sg.p1; pb += 32) {
      int blk = 0;
      if (pb + lane < sg.p1) {
        blk = p.block_table[(size_t)(s / p.bt_div) * p.max_pages + pb + lane];
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

constexpr int THREADS = 384;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tc_pair_decode_kernel(const __grid_constant__ CUtensorMap tm_cache,
                          const __grid_constant__ CUtensorMap tm_q, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t rank = cluster_ctarank();  // 0: score CTA, 1: value CTA
  const uint32_t peer = rank ^ 1u;
  const uint32_t sbase = smem_u32(smem);
  Ctx cx;
  cx.bar0 = sbase + (rank == 0 ? S_OFF_BAR : V_OFF_BAR);
  cx.abort = reinterpret_cast<volatile int*>(smem + (rank == 0 ? S_OFF_ABORT : V_OFF_ABORT));
  cx.peer_abort = mapa_shared(sbase + (rank == 0 ? V_OFF_ABORT : S_OFF_ABORT), peer);
  cx.dev_status = p.dev_status;
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(smem + (rank == 0 ? S_OFF_TSLOT : V_OFF_TSLOT));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x >> 1;
  const WorkerPlan w = reinterpret_cast<const WorkerPlan*>(p.ws + p.L.workers)[g];
  const SeqPlan* seqs = reinterpret_cast<const SeqPlan*>(p.ws + p.L.seqs);
  // Swizzled operand tiles need 1024-byte alignment of the shared window.
  const bool aligned = (sbase & 1023u) == 0;

  if (threadIdx.x == 0) {
    if (rank == 0) {
      for (int i = 0; i < NKS; ++i) {
        mbar_init(cx.bar(KFULL + i), 1);
        mbar_init(cx.bar(KEMPTY + i), 4);  // page: 3 + the QK commit; Q half: 2 warps x 2
      }
      for (int i = 0; i < NSB; ++i) {
        mbar_init(cx.bar(SFULL + i), 1);
        mbar_init(cx.bar(SFREE + i), 4);
      }
      for (int i = 0; i < NP; ++i) mbar_init(cx.bar(PEMPTY + i), 1);
      mbar_init(cx.bar(QTMEM), 4);
      mbar_init(cx.bar(QEMPTY), NQK);  // one commit per QK issuer
      for (int i = 0; i < NQK; ++i) mbar_init(cx.bar(SFINAL + i), 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(cx.bar(MREADY + i), 4);
        mbar_init(cx.bar(LXREADY + i), 4);
      }
    } else {
      for (int i = 0; i < NVS; ++i) {
        mbar_init(cx.bar(VFULL + i), 1);
        mbar_init(cx.bar(VEMPTY + i), 1);
      }
      for (int i = 0; i < NP; ++i) {
        mbar_init(cx.bar(PFULL + i), 1);
        mbar_init(cx.bar(ODONE + i), 1);
        mbar_expect_tx(cx.bar(PFULL + i), P_TX);  // armed for the slot's first page
      }
      mbar_init(cx.bar(ORESC), 4);
      mbar_init(cx.bar(WORK), 1);
      mbar_init(cx.bar(EPI), 4);
      mbar_init(cx.bar(OFREE), 4);
      mbar_init(cx.bar(OFREE + 1), 4);
      mbar_init(cx.bar(VFINAL), 1);
    }
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
  const bool active = aligned && w.n_pages > 0;

  if (active && rank == 0) {
    // ============================================================ score CTA
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      // ring items in order: per sequence its two Q halves (rows 0-63,
      // 64-127 of Q_cat), then its pages
      if (lane == 0) {
        tma_prefetch_desc(&tm_cache);
        tma_prefetch_desc(&tm_q);
      }
      uint32_t rk = 0;  // ring items issued
      auto put = [&](const CUtensorMap* map, int y) -> bool {
#ifdef MLA_TEST_HOOKS
        if (p.withhold) return false;  // test build: withhold every ring item
#endif
        const uint32_t st = rk % NKS;
        if (!cx.wait(KEMPTY + st, ((rk / NKS) & 1) ^ 1)) return false;
        mbar_expect_tx(cx.bar(KFULL + st), KSTAGE);
        for (int c = 0; c < NCHUNK; ++c)
          tma_load_2d(sbase + S_OFF_K + st * KSTAGE + c * CHUNK, map, c * 64, y, cx.bar(KFULL + st));
        ++rk;
        return true;
      };
      const bool ok = for_each_page(
          p, w, seqs, g, lane, [&](uint32_t, int bk) -> bool { return put(&tm_cache, bk * PAGE); },
          [&](int s) -> bool { return put(&tm_q, s * NH) && put(&tm_q, s * NH + PAGE); });
      if (!ok && lane == 0) {  // let issued copies land before the CTA exits
        for (uint32_t k = rk > (uint32_t)NKS ? rk - NKS : 0; k < rk; ++k)
          mbar_wait_drain(cx.bar(KFULL + k % NKS), (k / NKS) & 1, DRAIN_NS);
      }
    } else if (warp == 1 || warp == 6) {
      // --------------------------------------------------------- QK issue
      // issuer e (warps 1, 6) takes the pages with it % 2 == e, into S
      // buffer e. Each waits for every sequence's Q (so none can fall a
      // phase behind) and arrives once per sequence on QEMPTY: by a commit
      // after its last QK of the sequence, or a plain arrive if it had none
      // (a commit with no new MMA since the thread's previous commit does not
      // arrive).
      if (lane == 0) {
        const uint32_t e = warp == 1 ? 0u : 1u;  // warp 7 has no role in the score CTA
        uint32_t it = 0, seg = 0;
        bool ok = true;
        for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
          Seg sg;
          if (!seg_at(w, seqs, g, s, sg)) continue;
          const int n = sg.p1 - sg.p0;
          ok = cx.wait(QTMEM, seg & 1);
          bool issued = false;
          for (int j = 0; ok && j < n; ++j, ++it) {
            if (it % NQK != e) continue;
            const uint32_t rk = it + 2 * (seg + 1);  // ring item: two Q halves per sequence so far
            const uint32_t st = rk % NKS, sb = it % NSB;
            ok = cx.wait(SFREE + sb, ((it / NSB) & 1) ^ 1) && cx.wait(KFULL + st, (rk / NKS) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t pg = sbase + S_OFF_K + st * KSTAGE;
#pragma unroll
            for (int kk = 0; kk < 4 * NCHUNK; ++kk)
              mma_ts(tmem + TM_S + sb * 64, tmem + TM_Q + kk * 8,
                     sdesc_sw128(pg + (kk >> 2) * CHUNK + (kk & 3) * 32, 16, 1024), IDESC_QK,
                     kk > 0 ? 1u : 0u);
            mbar_arrive_cnt(cx.bar(KEMPTY + st), 3);  // the commit brings the fourth
            mma_commit(cx.bar(KEMPTY + st));
            mma_commit(cx.bar(SFULL + sb));
            issued = true;
          }
          if (ok) {
            if (issued) mma_commit(cx.bar(QEMPTY));
            else mbar_arrive(cx.bar(QEMPTY));
          }
          ++seg;
        }
        if (!ok) {
          mma_commit(cx.bar(SFINAL + e));
          mbar_wait_drain(cx.bar(SFINAL + e), 0, DRAIN_NS);
        }
      }
    } else if ((warp >= 2 && warp <= 5) || (warp >= 8 && warp <= 11)) {
      // ---------------------------------------------------------- softmax
      // Two groups of four warps (G = 0: warps 2-5, G = 1: warps 8-11) take
      // the pages in turn, page it by group it % 2, so one group's
      // exponentials and P stores overlap the other's. Both use the same
      // reference maximum for every page: the group of page it reads the
      // reference page it - 1 used (published in shared memory) before it
      // fixes its own (the lazy rescale rule). Each group keeps l over its own
      // pages; at a sequence's end the group of the last page adds the other
      // group's l, brought to the final reference.
      const int G = warp >= 8 ? 1 : 0;
      const int q4 = warp & 3;
      const int row = q4 * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      const uint32_t peer_pfull0 = mapa_shared(sbase + V_OFF_BAR + 8u * PFULL, peer);
      const uint32_t peer_p0 = mapa_shared(sbase + V_OFF_P, peer);
      const uint32_t peer_x0 = mapa_shared(sbase + V_OFF_X, peer);
      float* lse_part = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.lse_part);
      const float c = p.scale_log2;
      float* mref = reinterpret_cast<float*>(smem + S_OFF_MREF);  // [2][NH]
      float* lxl = reinterpret_cast<float*>(smem + S_OFF_LX);     // [2][NH] l
      float* lxm = lxl + 2 * NH;                                  // [2][NH] its reference
      // This thread's Q_cat row from ring item rq (rows 0-63) or rq + 1
      // (rows 64-127), un-swizzled, into TMEM columns [TM_Q, TM_Q + 288);
      // the item's two warps then release it.
      auto load_q = [&](uint32_t rq) -> bool {
        const uint32_t k = rq + (uint32_t)(q4 >> 1), st = k % NKS;
        if (!__all_sync(0xffffffffu, cx.wait(KFULL + st, (k / NKS) & 1))) return false;
        const uint8_t* src = smem + S_OFF_K + st * KSTAGE + (row & 63) * 128;
        const int sw = row & 7;
#pragma unroll 3
        for (int c = 0; c < NCHUNK; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + c * CHUNK + ((u ^ sw) << 4));
            v[4 * u] = x.x;
            v[4 * u + 1] = x.y;
            v[4 * u + 2] = x.z;
            v[4 * u + 3] = x.w;
          }
          tmem_st32(lane_base + TM_Q + c * 32, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cnt(cx.bar(KEMPTY + st), 2);
          mbar_arrive(cx.bar(QTMEM));
        }
        return true;
      };
      uint32_t it = 0, seg = 0, nlx = 0;  // nlx: sequences so far with two or more pages
      Seg sg;
      bool have = next_seg(w, seqs, g, w.seq_begin, sg);
      bool ok = !have || G == 1 || load_q(0);
      for (; ok && have; ++seg) {
        Seg nx;
        const bool have_next = next_seg(w, seqs, g, sg.s + 1, nx);
        const int n = sg.p1 - sg.p0;
        const uint32_t rq_next = it + n + 2 * (seg + 1);  // ring item of the next sequence's Q
        float m_own = 0.f, l = 0.f;  // this group's last reference and its l relative to it
        bool mine = false;
        for (int j = 0; j < n; ++j, ++it) {
          if ((int)(it & 1u) != G) continue;
          const uint32_t sb = it % NSB;
          ok = __all_sync(0xffffffffu, cx.wait(SFULL + sb, (it / NSB) & 1));
          if (!ok) break;
          tc_fence_after();
          uint32_t sa[32], sc[32];
          tmem_ld32(lane_base + TM_S + sb * 64, sa);
          tmem_ld32(lane_base + TM_S + sb * 64 + 32, sc);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(cx.bar(SFREE + sb));

          const int nvalid = min(PAGE, sg.len - (sg.p0 + j) * PAGE);
          if (nvalid < PAGE) {  // ragged tail: -inf scores give p = 0
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (i >= nvalid) sa[i] = 0xff800000u;
              if (32 + i >= nvalid) sc[i] = 0xff800000u;
            }
          }
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            mx[0] = fmaxf(mx[0], __uint_as_float(sa[i]));
            mx[1] = fmaxf(mx[1], __uint_as_float(sa[i + 1]));
            mx[2] = fmaxf(mx[2], __uint_as_float(sc[i]));
            mx[3] = fmaxf(mx[3], __uint_as_float(sc[i + 1]));
          }
          const float mp = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c;
          // reference maximum of this page: the page maximum on a sequence's
          // first page, else the previous page's reference unless this page's
          // maximum exceeds it by more than 8 (then O is rescaled by alpha)
          float m_use = mp, alpha = 1.f;
          bool resc = false;
          if (j > 0) {
            const uint32_t pi = it - 1;  // the other group's page
            ok = __all_sync(0xffffffffu, cx.wait(MREADY + (pi & 1), (pi >> 1) & 1));
            if (!ok) break;
            const float m_prev = mref[(pi & 1) * NH + row];
            if (mp > m_prev + 8.f) {
              alpha = ex2_approx(m_prev - mp);
              resc = true;
            } else {
              m_use = m_prev;
            }
          }
          mref[(it & 1) * NH + row] = m_use;
          __syncwarp();
          if (lane == 0) mbar_arrive(cx.bar(MREADY + (it & 1)));

          const float nm = -m_use;
          float sm[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float e0 = ex2_approx(fmaf(__uint_as_float(sa[2 * i]), c, nm));
            const float e1 = ex2_approx(fmaf(__uint_as_float(sa[2 * i + 1]), c, nm));
            const float e2 = ex2_approx(fmaf(__uint_as_float(sc[2 * i]), c, nm));
            const float e3 = ex2_approx(fmaf(__uint_as_float(sc[2 * i + 1]), c, nm));
            sm[0] += e0;
            sm[1] += e1;
            sm[2] += e2;
            sm[3] += e3;
            pk[i] = pack_bf16x2(e0, e1);
            pk[16 + i] = pack_bf16x2(e2, e3);
          }
          const float sum = (sm[0] + sm[1]) + (sm[2] + sm[3]);
          // the references only grow, so the factor is at most 1
          l = mine ? fmaf(l, ex2_approx(m_own - m_use), sum) : sum;
          m_own = m_use;
          mine = true;
          const bool last = j == n - 1;
          float inv_l = 0.f, lse = 0.f;
          if (last) {
            float lt = l;
            if (n >= 2) {  // the other group's pages of this sequence
              ok = __all_sync(0xffffffffu, cx.wait(LXREADY + (nlx & 1), (nlx >> 1) & 1));
              if (!ok) break;
              lt = fmaf(lxl[(nlx & 1) * NH + row], ex2_approx(lxm[(nlx & 1) * NH + row] - m_use), l);
            }
            inv_l = 1.f / lt;
            lse = (m_use + log2f(lt)) * 0.69314718055994531f;
          } else if (j == n - 2) {  // this group's last page of the sequence
            lxl[(nlx & 1) * NH + row] = l;
            lxm[(nlx & 1) * NH + row] = m_use;
            __syncwarp();
            if (lane == 0) mbar_arrive(cx.bar(LXREADY + (nlx & 1)));
          }

          // P row (and the row's rescale factor, 1 / l on the last page)
          // straight into P slot it % NP of the value CTA
          const uint32_t slot = it % NP;
          ok = __all_sync(0xffffffffu, cx.wait_cluster(PEMPTY + slot, ((it / NP) & 1) ^ 1));
          if (!ok) break;
          const uint32_t pf = peer_pfull0 + 8u * slot;
          const uint32_t prow = peer_p0 + slot * P_BYTES + row * 16;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            st_async_v4(prow + u * P_KGROUP, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3],
                        pf);
          const uint32_t px = peer_x0 + slot * X_BYTES;
          st_async_b32(px + XOFF_ALPHA + 4 * row, __float_as_uint(alpha), pf);
          st_async_b32(px + XOFF_INVL + 4 * row, __float_as_uint(inv_l), pf);
          const bool any_resc = __any_sync(0xffffffffu, resc);
          if (lane == 0) st_async_b32(px + XOFF_FLAG + 4 * q4, any_resc ? 1u : 0u, pf);
          if (last) {
            if (sg.slot < 0) p.lse[(size_t)sg.s * NH + row] = lse;
            else lse_part[(size_t)sg.slot * NH + row] = lse;
          }

          // the next sequence's Q as soon as this one's last QK is done (the
          // QK of its first page then overlaps the softmax of this last page)
          if (have_next && j == (n >= 2 ? n - 2 : 0)) {
            ok = __all_sync(0xffffffffu, cx.wait(QEMPTY, seg & 1));
            if (!ok) break;
            tc_fence_after();
            ok = load_q(rq_next);
            if (!ok) break;
          }
        }
        if (!ok) break;
        if (n >= 2) ++nlx;
        sg = nx;
        have = have_next;
      }
    }
  } else if (active) {
    // ============================================================ value CTA
    // O / l for column half `half` of a finished sequence (epilogue warps:
    // warp w owns rows [32 (w % 4), 32 (w % 4) + 32)). Per 32-column block
    // the thread of row r parks its 128 bytes in a swizzled staging tile,
    // then each store instruction writes 4 whole 128-byte row pieces; the
    // next block's TMEM load is in flight meanwhile. Arrives on OFREE + half.
    auto write_half = [&](const Seg& sg, int half, float inv_l) {
      const int q4 = warp & 3;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)half * (DC / 2);
      uint8_t* stg = smem + V_OFF_STG + (warp - 2) * 32 * 128;
      if (sg.slot >= 0) {
        // a split partial, in bf16: per two 32-column blocks the thread of
        // row r parks its 64 values (128 bytes) in the staging tile, then
        // each store instruction writes 4 whole 128-byte row pieces
        __nv_bfloat16* d16 = reinterpret_cast<__nv_bfloat16*>(const_cast<char*>(p.ws) + p.L.o_part) +
                             (size_t)sg.slot * NH * DC + half * (DC / 2);
#pragma unroll 1
        for (int cc = 0; cc < HALF_BLOCKS; cc += 2) {
          uint32_t va[32], vb[32];
          tmem_ld32(lane_base + cc * 32, va);
          tmem_ld32(lane_base + (cc + 1) * 32, vb);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t* v = (u < 4 ? va : vb) + 8 * (u & 3);
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((u ^ (lane & 7)) << 4)) = make_uint4(
                pack_bf16x2(__uint_as_float(v[0]) * inv_l, __uint_as_float(v[1]) * inv_l),
                pack_bf16x2(__uint_as_float(v[2]) * inv_l, __uint_as_float(v[3]) * inv_l),
                pack_bf16x2(__uint_as_float(v[4]) * inv_l, __uint_as_float(v[5]) * inv_l),
                pack_bf16x2(__uint_as_float(v[6]) * inv_l, __uint_as_float(v[7]) * inv_l));
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3), u = lane & 7;
            const uint4 x = *reinterpret_cast<const uint4*>(stg + r * 128 + ((u ^ (r & 7)) << 4));
            *reinterpret_cast<uint4*>(d16 + (size_t)(q4 * 32 + r) * DC + cc * 32 + 8 * u) = x;
          }
          __syncwarp();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(OFREE + half));
        return;
      }
      // the final o_lat of an unsplit sequence, in fp32
      float* dst0 = p.o_lat + (size_t)sg.s * NH * DC + half * (DC / 2);
      auto put_block = [&](int cc, const uint32_t (&v)[32]) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<float4*>(stg + lane * 128 + ((u ^ (lane & 7)) << 4)) =
              make_float4(__uint_as_float(v[4 * u]) * inv_l, __uint_as_float(v[4 * u + 1]) * inv_l,
                          __uint_as_float(v[4 * u + 2]) * inv_l,
                          __uint_as_float(v[4 * u + 3]) * inv_l);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3), u = lane & 7;
          const float4 x = *reinterpret_cast<const float4*>(stg + r * 128 + ((u ^ (r & 7)) << 4));
          *reinterpret_cast<float4*>(dst0 + (size_t)(q4 * 32 + r) * DC + cc * 32 + 4 * u) = x;
        }
        __syncwarp();
      };
      uint32_t va[32], vb[32];
      tmem_ld32(lane_base, va);
#pragma unroll 1
      for (int cc = 0; cc < HALF_BLOCKS; cc += 2) {
        tmem_ld_wait();
        tmem_ld32(lane_base + (cc + 1) * 32, vb);
        put_block(cc, va);
        tmem_ld_wait();
        if (cc + 2 < HALF_BLOCKS) tmem_ld32(lane_base + (cc + 2) * 32, va);
        put_block(cc + 1, vb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(OFREE + half));
    };
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0) tma_prefetch_desc(&tm_cache);
      uint32_t issued = 0;
      const bool ok = for_each_page(
          p, w, seqs, g, lane,
          [&](uint32_t k, int bk) -> bool {
            const uint32_t st = k % NVS;
            if (!cx.wait(VEMPTY + st, ((k / NVS) & 1) ^ 1)) return false;
            mbar_expect_tx(cx.bar(VFULL + st), VSTAGE);
            for (int c = 0; c < VCHUNK; ++c)
              tma_load_2d(sbase + V_OFF_V + st * VSTAGE + c * CHUNK, &tm_cache, c * 64, bk * PAGE,
                          cx.bar(VFULL + st));
            issued = k + 1;
            return true;
          },
          [](int) { return true; });
      if (!ok && lane == 0) {
        for (uint32_t k = issued > (uint32_t)NVS ? issued - NVS : 0; k < issued; ++k)
          mbar_wait_drain(cx.bar(VFULL + k % NVS), (k / NVS) & 1, DRAIN_NS);
      }
    } else if (warp == 1) {
      // --------------------------------------------------------- PV issue
      if (lane == 0) {
        uint32_t it = 0, seg = 0, nres = 0;
        bool ok = true;
        // 128 floats of a P slot's extras into a private copy
        auto copy_rows = [&](uint32_t dst_off, const uint8_t* src) {
#pragma unroll 4
          for (int i = 0; i < NH / 4; ++i)
            reinterpret_cast<uint4*>(smem + dst_off)[i] = reinterpret_cast<const uint4*>(src)[i];
        };
        // a command for epilogue group 0: kind 1 rescale before page it,
        // kind 2 sequence finished with page it
        auto post = [&](uint32_t kind, uint32_t page) {
          volatile uint32_t* cmd = reinterpret_cast<volatile uint32_t*>(smem + V_OFF_CMD);
          cmd[0] = kind;
          cmd[1] = page;
          mbar_arrive(cx.bar(WORK));
        };
        for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
          Seg sg;
          if (!seg_at(w, seqs, g, s, sg)) continue;
          const int n = sg.p1 - sg.p0;
          for (int j = 0; ok && j < n; ++j, ++it) {
            const uint32_t vs = it % NVS, slot = it % NP;
            ok = cx.wait(VFULL + vs, (it / NVS) & 1) &&
                 cx.wait_cluster(PFULL + slot, (it / NP) & 1);
            if (!ok) break;
            mbar_expect_tx(cx.bar(PFULL + slot), P_TX);  // armed for the slot's next page
            const uint8_t* xs = smem + V_OFF_X + slot * X_BYTES;
            const uint32_t* xf = reinterpret_cast<const uint32_t*>(xs + XOFF_FLAG);
            if (xf[0] | xf[1] | xf[2] | xf[3]) {  // never on j == 0
              // rescale O by alpha (once PV of the previous page is done)
              copy_rows(V_OFF_XA, xs + XOFF_ALPHA);
              post(1u, it);
              ok = cx.wait(ORESC, nres & 1);
              ++nres;
              if (!ok) break;
            }
            if (j == n - 1)  // before the slot is freed
              copy_rows(V_OFF_XL + (seg & 1) * 4 * NH, xs + XOFF_INVL);
            tc_fence_after();
            const uint32_t pa = sbase + V_OFF_P + slot * P_BYTES;
            const uint32_t vb = sbase + V_OFF_V + vs * VSTAGE;
            auto pv = [&](int k, int h) {
              mma_ss(tmem + h * 256, sdesc_noswz(pa + k * 2 * P_KGROUP, P_KGROUP, 128),
                     sdesc_sw128(vb + h * 4 * CHUNK + k * 2048, CHUNK, 1024), IDESC_PV,
                     (j > 0 || k > 0) ? 1u : 0u);
            };
            if (j == 0 && seg > 0) {
              // a sequence's first page: column half h of O once the previous
              // sequence's half h has been written out
              for (int h = 0; ok && h < 2; ++h) {
                ok = cx.wait(OFREE + h, (seg - 1) & 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k) pv(k, h);
              }
              if (!ok) break;
            } else {
              // alternate the two accumulators so consecutive products are
              // independent
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                pv(k, 0);
                pv(k, 1);
              }
            }
            mma_commit(cx.bar(VEMPTY + vs));
            mma_commit(cx.bar(ODONE + slot));
            mma_commit_mc(sbase + S_OFF_BAR + 8u * (PEMPTY + slot), 1u);  // the score CTA's slot barrier
            if (j == n - 1) post(2u, it);  // sequence finished
          }
          ++seg;
        }
        if (!ok) {
          mma_commit(cx.bar(VFINAL));
          mbar_wait_drain(cx.bar(VFINAL), 0, DRAIN_NS);
        }
      }
    } else if (warp >= 2 && warp <= 5) {
      // ------------------------------------------------ epilogue, group 0
      // Sleeps until the issuer posts a command: rescale O (all 512
      // columns) by alpha once PV of the page before is done, or, at a
      // sequence's end, start group 1 and write O columns [0, 256).
      const int q4 = warp & 3;
      const int row = q4 * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      const volatile uint32_t* cmd = reinterpret_cast<const volatile uint32_t*>(smem + V_OFF_CMD);
      int nseg = 0;
      for (int s = w.seq_begin; s <= w.seq_end; ++s) {
        Seg sg;
        if (seg_at(w, seqs, g, s, sg)) ++nseg;
      }
      Seg sg;
      bool ok = nseg == 0 || next_seg(w, seqs, g, w.seq_begin, sg);
      uint32_t ncmd = 0;
      for (int done = 0; ok && done < nseg;) {
        ok = __all_sync(0xffffffffu, cx.wait_sleepy(WORK, ncmd & 1));
        if (!ok) break;
        ++ncmd;
        const uint32_t kind = cmd[0], page = cmd[1];
        const uint32_t pd = kind == 1u ? page - 1 : page;  // page whose PV must be done
        ok = __all_sync(0xffffffffu, cx.wait(ODONE + pd % NP, (pd / NP) & 1));
        if (!ok) break;
        tc_fence_after();
        if (kind == 1u) {
          const float alpha = reinterpret_cast<const float*>(smem + V_OFF_XA)[row];
#pragma unroll 1
          for (int cc = 0; cc < DC / 32; ++cc) {
            uint32_t v[32];
            tmem_ld32(lane_base + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(lane_base + cc * 32, v);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(cx.bar(ORESC));
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(cx.bar(EPI));
          write_half(sg, 0, reinterpret_cast<const float*>(smem + V_OFF_XL + (done & 1) * 4 * NH)[row]);
          ++done;
          if (done < nseg) ok = next_seg(w, seqs, g, sg.s + 1, sg);
        }
      }
    } else if (warp >= 6 && warp <= 9) {
      // ------------------------------------------------ epilogue, group 1
      // At each sequence's end: O columns [256, 512).
      const int row = (warp & 3) * 32 + lane;
      const float* xl = reinterpret_cast<const float*>(smem + V_OFF_XL);
      uint32_t seg = 0;
      bool ok = true;
      for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
        Seg sg;
        if (!seg_at(w, seqs, g, s, sg)) continue;
        ok = __all_sync(0xffffffffu, cx.wait_sleepy(EPI, seg & 1));
        if (!ok) break;
        tc_fence_after();
        write_half(sg, 1, xl[(seg & 1) * NH + row]);
        ++seg;
      }
    }
  }
  __syncthreads();
  if (*cx.abort) {
    // stores this CTA sent to the peer complete on the peer's barriers; give
    // any still in flight time to land before the cluster may exit
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  cluster_sync_all();  // neither CTA leaves while the peer may still access it
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

// A [rows][576] bf16 array (the paged cache, or Q_cat) as 2-D tiles of 64
// rows x 64 columns with 128-byte swizzle.
cudaError_t make_cache_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return cudaErrorMisalignedAddress;
  const cuuint64_t dims[2] = {(cuuint64_t)ROW, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ROW * 2};
  const cuuint32_t box[2] = {64, PAGE};
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
  static unsigned long long smem_done = 0;
  if (set_max_smem_once((const void*)tc_pair_decode_kernel, (int)SMEM_BYTES, smem_done) != cudaSuccess)
    return 0;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2 > 0 ? sms / 2 : 1));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  int n = 0;
  // The kernel's cluster shape is fixed at compile time; some runtimes also
  // want it in the launch configuration.
  if (cudaOccupancyMaxActiveClusters(&n, tc_pair_decode_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, tc_pair_decode_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
  }
  cached[dev] = n;
  have[dev] = true;
  return n;
}

}  // namespace tcp

int tc_pair_workers(int sms) {
  int n = sms / 2 > 0 ? sms / 2 : 1;
  const int mc = tcp::max_clusters();
  if (mc > 0 && mc < n) n = mc;
  return n;
}

cudaError_t tc_pair_launch(const void* q_cat, const void* cache, const int32_t* block_table,
                           int max_pages, int num_pages, int B, int workers, float scale,
                           const void* ws, const WorkspaceLayout& L, float* o_lat, float* lse,
                           int32_t* dev_status, int bt_div, cudaStream_t s) {
  CUtensorMap tm_cache, tm_q;
  cudaError_t e = tcp::make_cache_map(&tm_cache, cache, (uint64_t)num_pages * tcp::PAGE);
  if (e != cudaSuccess) return e;
  // Q_cat [B * 128][576] has the cache's row shape: the same tiling
  e = tcp::make_cache_map(&tm_q, q_cat, (uint64_t)B * tcp::NH);
  if (e != cudaSuccess) return e;
  tcp::Params p;
  p.block_table = block_table;
  p.ws = reinterpret_cast<const char*>(ws);
  p.L = L;
  p.o_lat = o_lat;
  p.lse = lse;
  p.dev_status = dev_status;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.bt_div = bt_div > 0 ? bt_div : 1;
  p.withhold = g_test_withhold;
  static unsigned long long smem_done = 0;
  e = set_max_smem_once((const void*)tcp::tc_pair_decode_kernel, (int)tcp::SMEM_BYTES, smem_done);
  if (e != cudaSuccess) return e;
  tcp::tc_pair_decode_kernel<<<2 * workers, tcp::THREADS, tcp::SMEM_BYTES, s>>>(tm_cache, tm_q, p);
  return cudaGetLastError();
}

}  // namespace mla
