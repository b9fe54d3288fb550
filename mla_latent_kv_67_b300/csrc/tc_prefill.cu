// Prefill in the MHA form: the latent cache rows of a prompt are expanded to
// per-head keys and values once, then causal attention runs over them on the
// 5th-generation tensor cores ("kv-cache 的优化学习", closing note: the cache
// is stored in the MLA form, expanded to MHA for prefill and kept latent for
// decode; "DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现",
// 2.1: k^C = W^UK c, v^C = W^UV c, and 3.2: the key is [k^C_h ; k^R] with
// the RoPE key shared by all heads; the absorbed form is an inference-time
// rewrite for decoding).
//
//   q      [N][n_h][d_h + d_R]   (RoPE already applied to the last d_R)
//   k_nope [N][n_h][d_h]         = c W^UK_h^T
//   rows   [N][d_c + d_R]        the latent rows; k_R = rows[:, d_c:]
//   v      [N][n_h][d_v]         = c W^UV_h^T
//   o_i,h  = sum_{j <= i} softmax_j(q_i,h . [k_nope_j,h ; k_R,j] * scale) v_j,h
//
// One CTA per (head, 128-query tile); heads in groups of eight, the heaviest
// tiles (most keys) of a group first.
// Per 128-key tile: S = Q . K^T (M = 128 queries, N = 128 keys, K = 192)
// into one of two TMEM buffers, online softmax by four warps (thread = query
// row = TMEM lane; lazy rescale of O: only when a row maximum grows by more
// than 8 in log2 units, P and l using the same stale maximum), P as bf16 into
// TMEM, O += P . V (M = 128, N = d_v = 128, K = 128 keys). The diagonal tile
// masks keys after the query. Warp 0 streams the key/value tiles with TMA
// (two stages; a stage's keys are refilled once its S is done, its values
// once its PV is done, so the next keys do not wait for the PV), warp 1
// issues the S products and warp 6 the P.V products (one issuing thread
// reaches only about half the tensor core's rate at these shapes; two
// share it). Every wait is bounded and reports MLA_DEV_TIMEOUT.
#include <cudaTypedefs.h>
#include <math.h>

#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_decode.h"

namespace mla {
namespace tpf {

using namespace ptx;

constexpr int NH = 128, DH = 128, DR = 64, DC = 512, DV = 128, QW = DH + DR, ROW = DC + DR;
constexpr int HG = 8;  // heads per scheduling group
static_assert(NH % HG == 0, "head groups");
constexpr int TQ = 128, TK = 128;          // queries / keys per tile
constexpr uint32_t CH = 128 * 128;         // one 64-column chunk of a 128-row tile: 16 KB
constexpr int NQC = QW / 64;               // Q chunks: 3 (two no-PE, one RoPE)
constexpr int NVC = DV / 64;               // V chunks: 2
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t KSTAGE = (NQC + NVC) * CH;  // K (3 chunks) + V (2 chunks): 80 KB
constexpr int NST = 2;
constexpr uint32_t OFF_K = OFF_Q + NQC * CH;
enum {
  QFULL = 0,
  KFULL = 1,            // [NST] the tile's keys landed
  VFULL = KFULL + NST,  // [NST] the tile's values landed
  VEMPTY = VFULL + NST, // [NST] the tile's PV done (commit); its S done is SFULL
  SFULL = VEMPTY + NST, // [2]
  SFREE = SFULL + 2,    // [2] (4 warps)
  PFULL = SFREE + 2,    // [2] (4 warps)
  PFREE = PFULL + 2,    // [2] (commit)
  FIN = PFREE + 2,      // drain after an abort: S issuer
  FIN2 = FIN + 1,       // ... and PV issuer
  NBAR = FIN2 + 1
};
constexpr uint32_t OFF_BAR = OFF_K + NST * KSTAGE;
constexpr uint32_t OFF_TSLOT = OFF_BAR + 8 * NBAR;
constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");

// TMEM: S0 S1 (128 columns each) | O (128) | P0 P1 (64 each)
constexpr uint32_t TM_S = 0, TM_O = 256, TM_P = 384, TM_COLS = 512;
constexpr uint32_t IDESC_S = idesc_bf16_f32(TQ, TK, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(TQ, DV, false, true);
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_NS = 100000000ull;
constexpr int THREADS = 224;

struct Params {
  int N;                // tokens
  int n_qt;             // query tiles
  float scale_log2;
  __nv_bfloat16* o;     // [N][n_h][d_v]
  float* lse;           // [N][n_h] or null
  int32_t* dev_status;
};

__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile int* abort,
                                      int32_t* st) {
  return mbar_wait_bounded(bar, parity, abort, st, WAIT_NS);
}

__global__ void __launch_bounds__(THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_v,
                   const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Heads in groups of HG; within a group the heaviest query tiles (most key
  // tiles) first. The CTAs in flight then share the keys of a few heads,
  // which stay in L2, instead of touching the keys of every head at once.
  const int grp = (int)blockIdx.x / (HG * p.n_qt), r = (int)blockIdx.x % (HG * p.n_qt);
  const int h = grp * HG + r % HG;
  const int qt = p.n_qt - 1 - r / HG;
  const int q0 = qt * TQ;
  const int nkt = qt + 1;  // key tiles 0 .. qt

  if (threadIdx.x == 0) {
    mbar_init(bar(QFULL), 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(KFULL + i), 1);
      mbar_init(bar(VFULL + i), 1);
      mbar_init(bar(VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SFULL + i), 1);
      mbar_init(bar(SFREE + i), 4);
      mbar_init(bar(PFULL + i), 4);
      mbar_init(bar(PFREE + i), 1);
    }
    mbar_init(bar(FIN), 1);
    mbar_init(bar(FIN2), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tslot), TM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_kr);
    tma_prefetch_desc(&tm_v);
    mbar_expect_tx(bar(QFULL), NQC * CH);
    for (int c = 0; c < NQC; ++c) tma_load_3d(sb + OFF_Q + c * CH, &tm_q, 64 * c, h, q0, bar(QFULL));
    // A stage's keys and values are refilled separately: the keys of tile
    // kt + 2 as soon as S of tile kt is done, the values once its PV is
    // done. Keys run one tile ahead of values: K(kt + 1), then V(kt).
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    auto load_k = [&](int kt) -> bool {
      const int st = kt % NST;
      if (kt >= NST && !wait1(bar(SFULL + (kt & 1)), ((kt - NST) >> 1) & 1, abort_flag, p.dev_status))
        return false;
      const uint32_t dst = sb + OFF_K + st * KSTAGE;
      mbar_expect_tx(bar(KFULL + st), NQC * CH);
      tma_load_3d(dst, &tm_k, 0, h, kt * TK, bar(KFULL + st));
      tma_load_3d(dst + CH, &tm_k, 64, h, kt * TK, bar(KFULL + st));
      tma_load_2d(dst + 2 * CH, &tm_kr, DC, kt * TK, bar(KFULL + st));
      k_issued = kt + 1;
      return true;
    };
    auto load_v = [&](int kt) -> bool {
      const int st = kt % NST;
      if (!wait1(bar(VEMPTY + st), ((kt / NST) & 1) ^ 1, abort_flag, p.dev_status)) return false;
      const uint32_t dst = sb + OFF_K + st * KSTAGE + NQC * CH;
      mbar_expect_tx(bar(VFULL + st), NVC * CH);
      tma_load_3d(dst, &tm_v, 0, h, kt * TK, bar(VFULL + st));
      tma_load_3d(dst + CH, &tm_v, 64, h, kt * TK, bar(VFULL + st));
      v_issued = kt + 1;
      return true;
    };
    ok = load_k(0);
    for (int kt = 0; ok && kt < nkt; ++kt) {
      if (kt + 1 < nkt) ok = load_k(kt + 1);
      if (ok) ok = load_v(kt);
    }
    for (int i = k_issued > NST ? k_issued - NST : 0; i < k_issued; ++i)
      mbar_wait_drain(bar(KFULL + i % NST), (i / NST) & 1, DRAIN_NS);
    for (int i = v_issued > NST ? v_issued - NST : 0; i < v_issued; ++i)
      mbar_wait_drain(bar(VFULL + i % NST), (i / NST) & 1, DRAIN_NS);
    mbar_wait_drain(bar(QFULL), 0, DRAIN_NS);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------- S issue
    // S of key tile kt into S buffer kt & 1; the P.V products come from
    // warp 6, so the two chains share the tensor pipe instead of taking
    // turns in one issuing thread
    bool ok = wait1(bar(QFULL), 0, abort_flag, p.dev_status);
    bool any = false;
    for (int kt = 0; ok && kt < nkt; ++kt) {
      const int st = kt % NST, sbuf = kt & 1;
      ok = wait1(bar(SFREE + sbuf), ((kt >> 1) & 1) ^ 1, abort_flag, p.dev_status) &&
           wait1(bar(KFULL + st), (kt / NST) & 1, abort_flag, p.dev_status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t kt_base = sb + OFF_K + st * KSTAGE;
#pragma unroll
      for (int c = 0; c < NQC; ++c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + TM_S + sbuf * TK, sdesc_sw128(sb + OFF_Q + c * CH + kk * 32, 16, 1024),
                 sdesc_sw128(kt_base + c * CH + kk * 32, 16, 1024), IDESC_S, (c | kk) ? 1u : 0u);
      mma_commit(bar(SFULL + sbuf));
      any = true;
    }
    if (!ok && any) {
      mma_commit(bar(FIN));
      mbar_wait_drain(bar(FIN), 0, DRAIN_NS);
    }
  } else if (warp == 6 && lane == 0) {
    // ------------------------------------------------------------ PV issue
    bool ok = true, any = false;
    for (int kt = 0; ok && kt < nkt; ++kt) {
      const int st = kt % NST, pb = kt & 1;
      ok = wait1(bar(PFULL + pb), (kt >> 1) & 1, abort_flag, p.dev_status) &&
           wait1(bar(VFULL + st), (kt / NST) & 1, abort_flag, p.dev_status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t vt = sb + OFF_K + st * KSTAGE + NQC * CH;
#pragma unroll
      for (int kk = 0; kk < TK / 16; ++kk)
        mma_ts(tmem + TM_O, tmem + TM_P + pb * 64 + kk * 8, sdesc_sw128(vt + kk * 2048, CH, 1024),
               IDESC_PV, (kt > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar(PFREE + pb));
      mma_commit(bar(VEMPTY + st));
      any = true;
    }
    if (!ok && any) {
      mma_commit(bar(FIN2));
      mbar_wait_drain(bar(FIN2), 0, DRAIN_NS);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------- softmax
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int qi = q0 + row;  // this thread's query
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int kt = 0; kt < nkt; ++kt) {
      const int sbuf = kt & 1, pb = kt & 1;
      bool w = true;
      if (lane == 0) w = wait1(bar(SFULL + sbuf), (kt >> 1) & 1, abort_flag, p.dev_status);
      ok = __shfl_sync(0xffffffffu, w, 0);
      if (!ok) break;
      mbar_try_wait(bar(SFULL + sbuf), (kt >> 1) & 1);
      tc_fence_after();
      float s[TK];
#pragma unroll
      for (int b = 0; b < TK / 32; ++b) {
        uint32_t v[32];
        tmem_ld32(lane_base + TM_S + sbuf * TK + b * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * b + i] = __uint_as_float(v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SFREE + sbuf));
      // causal and length mask: key k0 + j is visible to query qi if
      // k0 + j <= qi and k0 + j < N
      const int k0 = kt * TK;
      const int lim = min(qi - k0, p.N - 1 - k0);  // last visible j
      if (lim < TK - 1) {
#pragma unroll
        for (int j = 0; j < TK; ++j)
          if (j > lim) s[j] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < TK; ++j) mx = fmaxf(mx, s[j]);
      const float mp = mx * c;
      float m_use = m, alpha = 1.f;
      bool resc = false;
      if (kt == 0) {
        m_use = mp;
      } else if (mp > m + 8.f) {
        m_use = mp;
        alpha = ex2_approx(m - mp);
        resc = true;
      }
      // a query row past the end of the prompt sees no key: keep it finite
      if (m_use == -INFINITY) m_use = 0.f;
      const float nm = -m_use;
      float sum = 0.f;
      uint32_t pk[TK / 2];
#pragma unroll
      for (int j = 0; j < TK / 2; ++j) {
        const float e0 = ex2_approx(fmaf(s[2 * j], c, nm));
        const float e1 = ex2_approx(fmaf(s[2 * j + 1], c, nm));
        sum += e0 + e1;
        pk[j] = pack_bf16x2(e0, e1);
      }
      l = (kt == 0) ? sum : fmaf(l, alpha, sum);
      m = m_use;
      if (__any_sync(0xffffffffu, resc)) {
        // this warp's rows of O, once the PV of the previous tile is done
        const int pi = kt - 1;
        bool w2 = true;
        if (lane == 0) w2 = wait1(bar(PFREE + (pi & 1)), (pi >> 1) & 1, abort_flag, p.dev_status);
        ok = __shfl_sync(0xffffffffu, w2, 0);
        if (!ok) break;
        mbar_try_wait(bar(PFREE + (pi & 1)), (pi >> 1) & 1);
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(lane_base + TM_O + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(lane_base + TM_O + cc * 32, v);
        }
        tmem_st_wait();
      }
      // P into TMEM buffer pb once the PV that last read it is done
      bool w3 = true;
      if (lane == 0) w3 = wait1(bar(PFREE + pb), ((kt >> 1) & 1) ^ 1, abort_flag, p.dev_status);
      ok = __shfl_sync(0xffffffffu, w3, 0);
      if (!ok) break;
      mbar_try_wait(bar(PFREE + pb), ((kt >> 1) & 1) ^ 1);
      tc_fence_after();
      uint32_t p0[32], p1[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        p0[j] = pk[j];
        p1[j] = pk[32 + j];
      }
      tmem_st32(lane_base + TM_P + pb * 64, p0);
      tmem_st32(lane_base + TM_P + pb * 64 + 32, p1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(PFULL + pb));
    }
    if (ok) {
      // O / l once the last PV is done
      const int last = nkt - 1;
      bool w = true;
      if (lane == 0) w = wait1(bar(PFREE + (last & 1)), (last >> 1) & 1, abort_flag, p.dev_status);
      ok = __shfl_sync(0xffffffffu, w, 0);
      if (ok) {
        mbar_try_wait(bar(PFREE + (last & 1)), (last >> 1) & 1);
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        // every lane runs the TMEM loads (warp-wide instructions); only rows
        // inside the prompt store
        const bool live = qi < p.N;
        __nv_bfloat16* dst = p.o + ((size_t)(live ? qi : 0) * NH + h) * DV;
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(lane_base + TM_O + cc * 32, v);
          tmem_ld_wait();
          uint32_t pkd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
          if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<uint4*>(dst + cc * 32)[i] =
                  make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
          }
        }
        if (live && p.lse) p.lse[(size_t)qi * NH + h] = (m + log2f(l)) * 0.69314718055994531f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
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

}  // namespace tpf

bool tc_prefill_supported(int n_h, int d_h, int d_r, int d_c, int d_v) {
  return n_h == tpf::NH && d_h == tpf::DH && d_r == tpf::DR && d_c == tpf::DC && d_v == tpf::DV &&
         tc_decode_supported(n_h, d_c, d_r, 64);
}

cudaError_t tc_prefill_launch(const void* q, const void* k_nope, const void* rows, const void* v,
                              void* o, float* lse, int N, float scale, int32_t* dev_status,
                              cudaStream_t s) {
  using namespace tpf;
  if (N <= 0) return cudaSuccess;
  CUtensorMap tm_q, tm_k, tm_kr, tm_v;
  cudaError_t e;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)QW, (cuuint64_t)NH, (cuuint64_t)N};
    const cuuint64_t str[2] = {(cuuint64_t)QW * 2, (cuuint64_t)NH * QW * 2};
    const cuuint32_t box[3] = {64, 1, TQ};
    if ((e = make_map(&tm_q, q, 3, dims, str, box)) != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)DH, (cuuint64_t)NH, (cuuint64_t)N};
    const cuuint64_t str[2] = {(cuuint64_t)DH * 2, (cuuint64_t)NH * DH * 2};
    const cuuint32_t box[3] = {64, 1, TK};
    if ((e = make_map(&tm_k, k_nope, 3, dims, str, box)) != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)ROW, (cuuint64_t)N};
    const cuuint64_t str[1] = {(cuuint64_t)ROW * 2};
    const cuuint32_t box[2] = {64, TK};
    if ((e = make_map(&tm_kr, rows, 2, dims, str, box)) != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)NH, (cuuint64_t)N};
    const cuuint64_t str[2] = {(cuuint64_t)DV * 2, (cuuint64_t)NH * DV * 2};
    const cuuint32_t box[3] = {64, 1, TK};
    if ((e = make_map(&tm_v, v, 3, dims, str, box)) != cudaSuccess) return e;
  }
  Params p;
  p.N = N;
  p.n_qt = (N + TQ - 1) / TQ;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.dev_status = dev_status;
  static unsigned long long smem_done = 0;
  e = set_max_smem_once((const void*)prefill_kernel, (int)SMEM_BYTES, smem_done);
  if (e != cudaSuccess) return e;
  prefill_kernel<<<p.n_qt * NH, THREADS, SMEM_BYTES, s>>>(tm_q, tm_k, tm_kr, tm_v, p);
  return cudaGetLastError();
}

}  // namespace mla
