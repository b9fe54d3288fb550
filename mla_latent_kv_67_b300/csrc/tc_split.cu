// tcgen05 decode attention over the paged latent cache with the latent
// dimension split across the two CTAs (two SMs) of a cluster (DeepSeek-V2
// shapes: 128 heads, d_c = 512, d_R = 64, 64-token pages, bf16).
//
// Per page the 128 heads of a sequence share every cached row, so the work
// is two dense products on the 5th-generation tensor cores
// ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现", 3.2: the
// score is the latent-space content part plus the RoPE part; the latent
// output is the probability-weighted sum of cached latents):
//   S = Q_cat . Page^T      M = 128 heads, N = 64 tokens,  K = 576
//   O += P . Page[:, 0:512] M = 128 heads, N = 512 latent, K = 64 tokens
// CTA r of the pair owns latent columns [256 r, 256 r + 256) -- its half of
// O (128 x 256 fp32, 256 TMEM columns) and of every page -- and rank 0 also
// owns the 64 RoPE columns. Each CTA reads only its columns of a page
// (40 KB / 32 KB instead of the whole 72 KB row block), computes the partial
// score S_r over its columns, and the two partials are exchanged through
// distributed shared memory (each CTA stores its partial in its own shared
// memory and loads the peer's; per page one remote arrival says "ours is
// ready" and one says "we have read yours"): both CTAs then hold
// S = S_0 + S_1, bit for bit the same, and run the same online softmax, so
// each can multiply the probabilities into its own half of O. At a sequence's end each CTA writes
// its own 128 KB of O, so the write-out of a split partial takes half as
// long as from one SM.
//
// Warps of each CTA (352 threads):
//   0-3   softmax: thread = head row = TMEM lane. Read S_r, exchange,
//         online softmax in log2 units with a lazy rescale (O is rescaled
//         only when a row's maximum grows by more than 8, i.e. a factor 256;
//         P and l use the same stale maximum, so the result is exact), P as
//         bf16 into TMEM for the PV product. Rank 0 also moves the
//         sequence's RoPE query columns into TMEM.
//   4-7   epilogue: at a sequence's end, O_r / l to global memory, while the
//         softmax warps carry on with the next sequence.
//   8     page producer: TMA of this CTA's columns of each page (3 stages).
//   9     S issuer: S_r = Q_r . Page_r^T (Q latent half from shared memory,
//         the RoPE query from TMEM), two S buffers; it also loads each
//         sequence's latent query half once the previous one is done with.
//   10    PV issuer: O_r += P . Page_r[:, latent] (P from TMEM, two buffers).
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
namespace tcs {

using namespace ptx;

constexpr int NH = 128, DC = 512, DR = 64, ROW = DC + DR, PAGE = 64;
constexpr int HALF = DC / 2;                // latent columns per CTA
constexpr int NLAT = HALF / 64;             // 64-column chunks of them: 4
constexpr uint32_t CHUNK = PAGE * 128;      // one chunk of a page: 64 tokens x 128 B
constexpr uint32_t QCHUNK = NH * 128;       // one chunk of Q: 128 heads x 128 B
constexpr int NKS = 3;                      // page stages
constexpr uint32_t KSTAGE = (NLAT + 1) * CHUNK;  // rank 0: latent + RoPE chunks
constexpr uint32_t XROW = 64 * 4;           // one row of an exchanged partial S

// shared memory
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + NLAT * QCHUNK;
constexpr uint32_t OFF_X = OFF_K + NKS * KSTAGE;
constexpr uint32_t OFF_L = OFF_X + NH * XROW;  // [2][NH] 1 / l of a finished sequence
enum {
  KFULL = 0,             // [NKS] page columns landed
  KEMPTY = NKS,          // [NKS] page consumed (PV commit)
  SFULL = 2 * NKS,       // [2] partial S written
  SFREE = SFULL + 2,     // [2] partial S read by the 4 softmax warps
  PFULL = SFREE + 2,     // [2] P written to TMEM (4 warps)
  PFREE = PFULL + 2,     // [2] PV that read the P buffer done (commit)
  QFULL = PFREE + 2,     // Q latent half of the sequence landed
  QFREE = QFULL + 1,     // last S of the sequence done (commit)
  QRREADY = QFREE + 1,   // RoPE query in TMEM (4 warps; rank 0)
  XREADY = QRREADY + 1,  // the peer's partial S is in its buffer (1 remote arrival)
  XFREE = XREADY + 1,    // the peer has read our partial S (1 remote arrival)
  XSTORED = XFREE + 1,   // our 4 softmax warps stored their rows of the partial S
  XREAD = XSTORED + 1,   // our 4 softmax warps read their rows of the peer's
  LREADY = XREAD + 1,    // [2] 1 / l of a sequence written (4 softmax warps)
  LFREE = LREADY + 2,    // [2] 1 / l read by the 4 epilogue warps
  ODONE = LFREE + 2,     // last PV of a sequence done (commit)
  OFREE = ODONE + 1,     // O written out (4 epilogue warps)
  FIN_S = OFREE + 1,     // drain after an abort (S issuer)
  FIN_P = FIN_S + 1,     // drain after an abort (PV issuer)
  NBAR = FIN_P + 1
};
constexpr uint32_t OFF_BAR = OFF_L + 2 * NH * 4;
constexpr uint32_t OFF_TSLOT = OFF_BAR + 8 * NBAR;
constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4;
static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
static_assert(OFF_K % 1024 == 0 && KSTAGE % 1024 == 0 && OFF_X % 16 == 0 && OFF_BAR % 8 == 0,
              "layout alignment");

// TMEM columns: O half | S0 S1 | P0 P1 | RoPE query (rank 0)
constexpr uint32_t TM_O = 0, TM_S = 256, TM_P = 384, TM_QR = 448, TM_COLS = 512;

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, HALF, false, true);
#ifdef MLA_TEST_HOOKS
constexpr uint64_t WAIT_NS = 20000000ull;  // test build: a withheld item times out in 20 ms
#else
constexpr uint64_t WAIT_NS = 2000000000ull;
#endif
constexpr uint64_t DRAIN_NS = 100000000ull;
constexpr int THREADS = 352;

struct Params {
  const int32_t* block_table;
  const char* ws;
  WorkspaceLayout L;
  const __nv_bfloat16* q_cat;
  float* o_lat;
  float* lse;
  int32_t* dev_status;
  int max_pages, num_pages;
  float scale_log2;
  int bt_div;    // new tokens per sequence: query row s uses block-table row s / bt_div
  int withhold;  // read by the test build only: the page producer issues nothing
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
  __device__ bool fail() const {
    st_cluster_u32(peer_abort, 1);
    return false;
  }
  // one thread polls
  __device__ bool wait(int i, uint32_t parity) const {
    return mbar_wait_bounded(bar(i), parity, abort, dev_status, WAIT_NS) || fail();
  }
  __device__ bool wait_cluster(int i, uint32_t parity) const {
    return mbar_wait_cluster_bounded(bar(i), parity, abort, dev_status, WAIT_NS) || fail();
  }
  __device__ bool wait_sleepy(int i, uint32_t parity) const {
    return mbar_wait_sleepy(bar(i), parity, abort, dev_status, WAIT_NS, 200) || fail();
  }
  // lane 0 of the warp polls; every lane then acquires the completed phase
  // itself (one try_wait each, which succeeds at once)
  __device__ bool warp_wait(int i, uint32_t parity, int lane) const {
    bool ok = true;
    if (lane == 0) ok = wait(i, parity);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar(i), parity);
    return ok;
  }
  __device__ bool warp_wait_cluster(int i, uint32_t parity, int lane) const {
    bool ok = true;
    if (lane == 0) ok = wait_cluster(i, parity);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait_cluster(bar(i), parity);
    return ok;
  }
  __device__ bool warp_wait_sleepy(int i, uint32_t parity, int lane) const {
    bool ok = true;
    if (lane == 0) ok = wait_sleepy(i, parity);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar(i), parity);
    return ok;
  }
};

// 16-byte read-only global load.
__device__ __forceinline__ uint4 ldg_nc_u4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
// 16-byte store to this CTA's shared memory.
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
// 16-byte load from another CTA's shared memory (cluster address from mapa).
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// 32-byte global store.
__device__ __forceinline__ void stg_v8(float* p, const float (&v)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]),
               "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tc_split_decode_kernel(const __grid_constant__ CUtensorMap tm_cache,
                           const __grid_constant__ CUtensorMap tm_q, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t rank = cluster_ctarank();
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
  const bool aligned = (sbase & 1023u) == 0;
  const int nchunk = rank == 0 ? NLAT + 1 : NLAT;  // page chunks this CTA loads

  if (threadIdx.x == 0) {
    for (int i = 0; i < NKS; ++i) {
      mbar_init(cx.bar(KFULL + i), 1);
      mbar_init(cx.bar(KEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(SFULL + i), 1);
      mbar_init(cx.bar(SFREE + i), 4);
      mbar_init(cx.bar(PFULL + i), 4);
      mbar_init(cx.bar(PFREE + i), 1);
      mbar_init(cx.bar(LREADY + i), 4);
      mbar_init(cx.bar(LFREE + i), 4);
    }
    mbar_init(cx.bar(QFULL), 1);
    mbar_init(cx.bar(QFREE), 1);
    mbar_init(cx.bar(QRREADY), 4);
    mbar_init(cx.bar(XREADY), 1);
    mbar_init(cx.bar(XFREE), 1);
    mbar_init(cx.bar(XSTORED), 4);
    mbar_init(cx.bar(XREAD), 4);
    mbar_init(cx.bar(ODONE), 1);
    mbar_init(cx.bar(OFREE), 4);
    mbar_init(cx.bar(FIN_S), 1);
    mbar_init(cx.bar(FIN_P), 1);
    *cx.abort = 0;
    if (!aligned) report(p.dev_status, MLA_DEV_TIMEOUT);
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  cluster_sync_all();  // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool active = aligned && w.n_pages > 0;

  if (active && warp < 4) {
    // ============================================================ softmax
    const int row = warp * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t peer_xrow = mapa_shared(sbase + OFF_X + row * XROW, peer);
    const uint32_t peer_xready = mapa_shared(cx.bar(XREADY), peer);
    const uint32_t peer_xfree = mapa_shared(cx.bar(XFREE), peer);
    const uint32_t my_xrow = sbase + OFF_X + row * XROW;
    const int xs = row & 15;  // 16-byte unit swizzle of the exchanged rows
    float* lse_part = reinterpret_cast<float*>(const_cast<char*>(p.ws) + p.L.lse_part);
    float* lbuf = reinterpret_cast<float*>(smem + OFF_L);
    const float c = p.scale_log2;
    // the RoPE query columns of sequence s, this thread's row, into registers
    uint4 qr[8];
    auto fetch_qr = [&](int s) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q_cat + ((size_t)s * NH + row) * ROW + DC);
#pragma unroll
      for (int u = 0; u < 8; ++u) qr[u] = ldg_nc_u4(src + u);
    };
    Seg sg;
    bool have = false;
    for (int s = w.seq_begin; s <= w.seq_end && !have; ++s) have = seg_at(w, seqs, g, s, sg);
    if (rank == 0 && have) fetch_qr(sg.s);
    uint32_t it = 0, seg = 0;
    bool ok = true;
    for (; ok && have; ++seg) {
      Seg nx;
      bool have_next = false;
      for (int s = sg.s + 1; s <= w.seq_end && !have_next; ++s) have_next = seg_at(w, seqs, g, s, nx);
      if (rank == 0) {
        // the S products of the previous sequence are done (its last S was
        // read below), so the RoPE query slot is free
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          v[4 * u] = qr[u].x;
          v[4 * u + 1] = qr[u].y;
          v[4 * u + 2] = qr[u].z;
          v[4 * u + 3] = qr[u].w;
        }
        tmem_st32(lane_base + TM_QR, v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(QRREADY));
      }
      float m = -INFINITY, l = 0.f;
      const int n = sg.p1 - sg.p0;
      for (int j = 0; j < n; ++j, ++it) {
        const uint32_t sb = it & 1u;
        // own partial S
        ok = cx.warp_wait(SFULL + sb, (it >> 1) & 1, lane);
        if (!ok) break;
        tc_fence_after();
        uint32_t sa[32], sc[32];
        tmem_ld32(lane_base + TM_S + sb * 64, sa);
        tmem_ld32(lane_base + TM_S + sb * 64 + 32, sc);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(SFREE + sb));
        // exchange: each CTA puts its partial in its own buffer (once the
        // peer has read the previous one) and reads the peer's from the
        // peer's buffer; per page only the 2 x 128 arrivals cross the pair,
        // every data byte is a plain store and a distributed shared load
        ok = cx.warp_wait_cluster(XFREE, (it & 1) ^ 1, lane);
        if (!ok) break;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          sts_v4(my_xrow + ((u ^ xs) << 4), sa[4 * u], sa[4 * u + 1], sa[4 * u + 2], sa[4 * u + 3]);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          sts_v4(my_xrow + (((8 + u) ^ xs) << 4), sc[4 * u], sc[4 * u + 1], sc[4 * u + 2],
                 sc[4 * u + 3]);
        // once all 128 rows are stored (each warp arrives on XSTORED), one
        // release arrival on the peer's barrier makes them visible to it
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(XSTORED));
        if (row == 0) {
          ok = cx.wait(XSTORED, it & 1);
          if (ok) mbar_arrive_remote(peer_xready);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ok = cx.warp_wait_cluster(XREADY, it & 1, lane);
        if (!ok) break;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = ld_cluster_v4(peer_xrow + ((u ^ xs) << 4));
          sa[4 * u] = __float_as_uint(__uint_as_float(sa[4 * u]) + __uint_as_float(x.x));
          sa[4 * u + 1] = __float_as_uint(__uint_as_float(sa[4 * u + 1]) + __uint_as_float(x.y));
          sa[4 * u + 2] = __float_as_uint(__uint_as_float(sa[4 * u + 2]) + __uint_as_float(x.z));
          sa[4 * u + 3] = __float_as_uint(__uint_as_float(sa[4 * u + 3]) + __uint_as_float(x.w));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = ld_cluster_v4(peer_xrow + (((8 + u) ^ xs) << 4));
          sc[4 * u] = __float_as_uint(__uint_as_float(sc[4 * u]) + __uint_as_float(x.x));
          sc[4 * u + 1] = __float_as_uint(__uint_as_float(sc[4 * u + 1]) + __uint_as_float(x.y));
          sc[4 * u + 2] = __float_as_uint(__uint_as_float(sc[4 * u + 2]) + __uint_as_float(x.z));
          sc[4 * u + 3] = __float_as_uint(__uint_as_float(sc[4 * u + 3]) + __uint_as_float(x.w));
        }
        // every row of the peer's buffer read (XREAD), then one arrival on
        // the peer's XFREE
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(XREAD));
        if (row == 0) {
          ok = cx.wait(XREAD, it & 1);
          if (ok) mbar_arrive_remote(peer_xfree);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;

        // online softmax (log2 units), both CTAs on the same S
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
        l = (j == 0) ? sum : fmaf(l, alpha, sum);
        m = m_use;

        if (__any_sync(0xffffffffu, resc)) {
          // rescale this warp's rows of O once the previous page's PV is done
          const uint32_t pi = it - 1;
          ok = cx.warp_wait(PFREE + (pi & 1), (pi >> 1) & 1, lane);
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
          tmem_st_wait();
        }
        // P into TMEM buffer it % 2 once the PV that last read it is done
        ok = cx.warp_wait(PFREE + sb, ((it >> 1) & 1) ^ 1, lane);
        if (!ok) break;
        tc_fence_after();
        tmem_st32(lane_base + TM_P + sb * 32, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.bar(PFULL + sb));
      }
      if (!ok) break;
      // sequence done: 1 / l for the epilogue warps (once they have read
      // the value of two sequences ago from the same slot), lse (rank 0)
      ok = cx.warp_wait(LFREE + (seg & 1), ((seg >> 1) & 1) ^ 1, lane);
      if (!ok) break;
      lbuf[(seg & 1) * NH + row] = 1.f / l;
      if (rank == 0) {
        const float lse = (m + log2f(l)) * 0.69314718055994531f;
        if (sg.slot < 0) p.lse[(size_t)sg.s * NH + row] = lse;
        else lse_part[(size_t)sg.slot * NH + row] = lse;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(LREADY + (seg & 1)));
      if (rank == 0 && have_next) fetch_qr(nx.s);  // the next sequence's RoPE query
      sg = nx;
      have = have_next;
    }
  } else if (active && warp == 8) {
    // ------------------------------------------------------- page producer
    if (lane == 0) tma_prefetch_desc(&tm_cache);
    uint32_t k = 0, issued = 0;  // pages walked, pages whose copies were issued
#ifdef MLA_TEST_HOOKS
    bool ok = !p.withhold;  // test build: withhold every page
#else
    bool ok = true;
#endif
    for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
      Seg sg;
      if (!seg_at(w, seqs, g, s, sg)) continue;
      for (int pb = sg.p0; ok && pb < sg.p1; pb += 32) {
        int blk = 0;
        if (pb + lane < sg.p1) {
          blk = p.block_table[(size_t)(s / p.bt_div) * p.max_pages + pb + lane];
          if (blk < 0 || blk >= p.num_pages) {
            report(p.dev_status, MLA_DEV_BAD_BLOCK);
            blk = 0;
          }
        }
        const int nb = min(32, sg.p1 - pb);
        for (int j = 0; ok && j < nb; ++j, ++k) {
          const int bk = __shfl_sync(0xffffffffu, blk, j);
          if (lane == 0) {
            const uint32_t st = k % NKS;
            ok = cx.wait(KEMPTY + st, ((k / NKS) & 1) ^ 1);
            if (ok) {
              mbar_expect_tx(cx.bar(KFULL + st), nchunk * CHUNK);
              const uint32_t dst = sbase + OFF_K + st * KSTAGE;
              for (int ch = 0; ch < nchunk; ++ch) {
                const int col = ch < NLAT ? HALF * (int)rank + 64 * ch : DC;
                tma_load_2d(dst + ch * CHUNK, &tm_cache, col, bk * PAGE, cx.bar(KFULL + st));
              }
              issued = k + 1;
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
    }
    if (!ok && lane == 0) {  // let issued copies land before the CTA exits
      for (uint32_t i = issued > (uint32_t)NKS ? issued - NKS : 0; i < issued; ++i)
        mbar_wait_drain(cx.bar(KFULL + i % NKS), (i / NKS) & 1, DRAIN_NS);
    }
  } else if (active && warp == 9) {
    // ------------------------------------------ S issuer and Q producer
    // The sequence's latent query half is loaded into the one Q buffer once
    // the previous sequence's last S products are done; the issuer has
    // nothing else to do meanwhile, so it issues that copy itself.
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      auto load_q = [&](int s) {
        mbar_expect_tx(cx.bar(QFULL), NLAT * QCHUNK);
        for (int ch = 0; ch < NLAT; ++ch)
          tma_load_2d(sbase + OFF_Q + ch * QCHUNK, &tm_q, HALF * (int)rank + 64 * ch, s * NH,
                      cx.bar(QFULL));
      };
      uint32_t it = 0, seg = 0;
      bool ok = true, any = false, q_pending = false;
      Seg sg;
      bool have = false;
      for (int s = w.seq_begin; s <= w.seq_end && !have; ++s) have = seg_at(w, seqs, g, s, sg);
      if (have) {
        load_q(sg.s);
        q_pending = true;
      }
      for (; ok && have; ++seg) {
        Seg nx;
        bool have_next = false;
        for (int s = sg.s + 1; s <= w.seq_end && !have_next; ++s) have_next = seg_at(w, seqs, g, s, nx);
        ok = cx.wait(QFULL, seg & 1);
        if (ok) q_pending = false;
        ok = ok && (rank != 0 || cx.wait(QRREADY, seg & 1));
        const int n = sg.p1 - sg.p0;
        for (int j = 0; ok && j < n; ++j, ++it) {
          const uint32_t st = it % NKS, sb = it & 1u;
          ok = cx.wait(SFREE + sb, ((it >> 1) & 1) ^ 1) && cx.wait(KFULL + st, (it / NKS) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t pg = sbase + OFF_K + st * KSTAGE;
          const uint32_t d = tmem + TM_S + sb * 64;
#pragma unroll
          for (int ch = 0; ch < NLAT; ++ch)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(d, sdesc_sw128(sbase + OFF_Q + ch * QCHUNK + kk * 32, 16, 1024),
                     sdesc_sw128(pg + ch * CHUNK + kk * 32, 16, 1024), IDESC_QK,
                     (ch | kk) != 0 ? 1u : 0u);
          if (rank == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(d, tmem + TM_QR + kk * 8, sdesc_sw128(pg + NLAT * CHUNK + kk * 32, 16, 1024),
                     IDESC_QK, 1u);
          }
          mma_commit(cx.bar(SFULL + sb));
          if (j == n - 1) mma_commit(cx.bar(QFREE));  // Q buffer free once these are done
          any = true;
        }
        if (!ok || !have_next) break;
        // the next sequence's Q into the buffer once this one's S products are done
        ok = cx.wait(QFREE, seg & 1);
        if (!ok) break;
        load_q(nx.s);
        q_pending = true;
        sg = nx;
      }
      if (q_pending) mbar_wait_drain(cx.bar(QFULL), seg & 1, DRAIN_NS);
      if (!ok && any) {
        mma_commit(cx.bar(FIN_S));
        mbar_wait_drain(cx.bar(FIN_S), 0, DRAIN_NS);
      }
    }
  } else if (active && warp == 10) {
    // ---------------------------------------------------------- PV issuer
    if (lane == 0) {
      uint32_t it = 0, seg = 0;
      bool ok = true, any = false;
      for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
        Seg sg;
        if (!seg_at(w, seqs, g, s, sg)) continue;
        const int n = sg.p1 - sg.p0;
        for (int j = 0; ok && j < n; ++j, ++it) {
          const uint32_t st = it % NKS, pb = it & 1u;
          ok = cx.wait(PFULL + pb, (it >> 1) & 1);
          if (ok && j == 0 && seg > 0) ok = cx.wait(OFREE, (seg - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t pg = sbase + OFF_K + st * KSTAGE;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + TM_O, tmem + TM_P + pb * 32 + kk * 8,
                   sdesc_sw128(pg + kk * 2048, CHUNK, 1024), IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(cx.bar(PFREE + pb));
          mma_commit(cx.bar(KEMPTY + st));
          if (j == n - 1) mma_commit(cx.bar(ODONE));
          any = true;
        }
        ++seg;
      }
      if (!ok && any) {
        mma_commit(cx.bar(FIN_P));
        mbar_wait_drain(cx.bar(FIN_P), 0, DRAIN_NS);
      }
    }
  } else if (active && warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ epilogue
    // O_r / l of a finished sequence: 8 blocks of 32 columns, each thread
    // (head row) storing its 128 contiguous bytes of a block with 32-byte
    // stores.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const float* lbuf = reinterpret_cast<const float*>(smem + OFF_L);
    __nv_bfloat16* o_part = reinterpret_cast<__nv_bfloat16*>(const_cast<char*>(p.ws) + p.L.o_part);
    uint32_t seg = 0;
    bool ok = true;
    for (int s = w.seq_begin; ok && s <= w.seq_end; ++s) {
      Seg sg;
      if (!seg_at(w, seqs, g, s, sg)) continue;
      ok = cx.warp_wait_sleepy(LREADY + (seg & 1), (seg >> 1) & 1, lane) &&
           cx.warp_wait_sleepy(ODONE, seg & 1, lane);
      if (!ok) break;
      tc_fence_after();
      const float inv_l = lbuf[(seg & 1) * NH + row];
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(LFREE + (seg & 1)));
      // the final o_lat row (fp32) of an unsplit sequence, else the bf16
      // partial slot
      const bool part = sg.slot >= 0;
      float* dst = p.o_lat + ((size_t)sg.s * NH + row) * DC + HALF * rank;
      __nv_bfloat16* d16 = o_part + ((size_t)(part ? sg.slot : 0) * NH + row) * DC + HALF * rank;
      auto put8 = [&](int col, const float (&v)[8]) {
        if (part)
          *reinterpret_cast<uint4*>(d16 + col) =
              make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                         pack_bf16x2(v[6], v[7]));
        else
          stg_v8(dst + col, v);
      };
      uint32_t va[32], vb[32];
      tmem_ld32(lane_base + TM_O, va);
#pragma unroll 1
      for (int cc = 0; cc < HALF / 32; cc += 2) {
        tmem_ld_wait();
        tmem_ld32(lane_base + TM_O + (cc + 1) * 32, vb);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(va[8 * q + e]) * inv_l;
          put8(cc * 32 + 8 * q, v);
        }
        tmem_ld_wait();
        if (cc + 2 < HALF / 32) tmem_ld32(lane_base + TM_O + (cc + 2) * 32, va);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(vb[8 * q + e]) * inv_l;
          put8((cc + 1) * 32 + 8 * q, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(OFREE));
      ++seg;
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
  if (warp == 8) {
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

// A [rows][576] bf16 array as 2-D tiles of `box_rows` rows x 64 columns with
// 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
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
  static unsigned long long smem_done = 0;
  if (set_max_smem_once((const void*)tc_split_decode_kernel, (int)SMEM_BYTES, smem_done) != cudaSuccess)
    return 0;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2 > 0 ? sms / 2 : 1));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  int n = 0;
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

int g_test_withhold = 0;  // set by the test build's mla_test_withhold_pages

cudaError_t tc_split_launch(const void* q_cat, const void* cache, const int32_t* block_table,
                            int max_pages, int num_pages, int B, int workers, float scale,
                            const void* ws, const WorkspaceLayout& L, float* o_lat, float* lse,
                            int32_t* dev_status, int bt_div, cudaStream_t s) {
  CUtensorMap tm_cache, tm_q;
  cudaError_t e = tcs::make_map(&tm_cache, cache, (uint64_t)num_pages * tcs::PAGE, tcs::PAGE);
  if (e != cudaSuccess) return e;
  e = tcs::make_map(&tm_q, q_cat, (uint64_t)B * tcs::NH, tcs::NH);
  if (e != cudaSuccess) return e;
  tcs::Params p;
  p.block_table = block_table;
  p.ws = reinterpret_cast<const char*>(ws);
  p.L = L;
  p.q_cat = reinterpret_cast<const __nv_bfloat16*>(q_cat);
  p.o_lat = o_lat;
  p.lse = lse;
  p.dev_status = dev_status;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.bt_div = bt_div > 0 ? bt_div : 1;
  p.withhold = g_test_withhold;
  static unsigned long long smem_done = 0;
  e = set_max_smem_once((const void*)tcs::tc_split_decode_kernel, (int)tcs::SMEM_BYTES, smem_done);
  if (e != cudaSuccess) return e;
  tcs::tc_split_decode_kernel<<<2 * workers, tcs::THREADS, tcs::SMEM_BYTES, s>>>(tm_cache, tm_q, p);
  return cudaGetLastError();
}

}  // namespace mla

#ifdef MLA_TEST_HOOKS
// Test build only: make the next decode launches' page producer withhold
// every page, so the bounded waits of both CTAs run out (20 ms in this
// build) and the kernel reports MLA_DEV_TIMEOUT and returns.
extern "C" void mla_test_withhold_pages(int on) { mla::g_test_withhold = on ? 1 : 0; }
#endif
