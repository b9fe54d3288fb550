// tcgen05 tile GEMM for the projections of a prompt (many tokens at once):
// the same products and epilogues as the weight-streaming GEMM of
// tc_gemm.cu ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现":
// 2.1 W^DKV with W^KR of 3.2 feeding the cache, 2.3 W^DQ and W^UQ with W^QR,
// and the expansion of cached latents through W^UK / W^UV of 2.1)
//
//   out[m][n] = sum_k X[m][k] W[n][k]     X [M][K] bf16 (tokens), W [N][K] bf16
//
// With thousands of tokens the product is bound by the tensor cores, not by
// the weight bytes, so the tile is the token side as the MMA's M (128 token
// rows) and 256 output features as N: D[128 tokens][256 features] in tensor
// memory, one 128 x 256 x 16 product per instruction. Persistent clusters of
// two CTAs (one per SM) walk pairs of tiles that share their 256 features
// (token tiles fastest, so the clusters in flight share a few weight tiles in
// L2); each CTA of a pair loads half of every weight chunk and multicasts it
// to both:
//   warp 0     TMA producer: X and W chunks of 64 along K into a 4-stage ring
//              (a stage is refilled once the products of both CTAs are done);
//   warp 1     MMA issuer: four products per chunk into one of two
//              accumulators (256 columns each), so the epilogue of a tile
//              overlaps the products of the next;
//   warps 2-5  epilogue: thread = token row = TMEM lane; reads its 256
//              features 32 at a time, applies the epilogue of tc_gemm.cu
//              (STORE, ROPE on the pairs of the RoPE columns, APPEND into the
//              paged cache row of the token) and stores its row piece.
// Every wait is bounded and reports MLA_DEV_TIMEOUT.
#include <cudaTypedefs.h>

#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_decode.h"

namespace mla {
namespace tg {

using namespace ptx;

constexpr int THREADS = 192;
constexpr int TM = 128;   // token rows per tile (MMA M)
constexpr int TN = 256;   // output features per tile (MMA N)
constexpr int NST = 4;    // ring stages
constexpr uint32_t A_BYTES = TM * 128;            // X chunk [128 rows][64 bf16]: 16 KB
constexpr uint32_t B_BYTES = TN * 128;            // W chunk [256 rows][64 bf16]: 32 KB
constexpr uint32_t STAGE = A_BYTES + B_BYTES;     // 48 KB
constexpr uint32_t OFF_BAR = NST * STAGE;
enum { FULL = 0, EMPTY = NST, TFULL = 2 * NST, TEMPTY = TFULL + 2, FIN = TEMPTY + 2, NBAR = FIN + 1 };
constexpr uint32_t OFF_TSLOT = OFF_BAR + 8 * NBAR;
constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;
constexpr uint32_t SMEM = OFF_ABORT + 4 + 1024;  // + alignment slack
constexpr uint32_t IDESC = idesc_bf16_f32(TM, TN, false, false);
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_NS = 100000000ull;

// 2-D tiled load global -> shared, written at the same shared offset in every
// CTA of `mask` in the cluster, completion counted on `bar` (same offset) in
// each of them.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(mask)
      : "memory");
}

struct Args {
  int M, N, K;
  int m_pairs, tiles;  // tiles: pairs of token tiles x feature tiles
  int vec;  // output rows take 16-byte stores (alignment checked on the host)
  int epi;
  void* out;
  long long ldo;
  int out_f32;
  const float* rope;
  int max_pos, d_r, rope_off, rope_period;
  const int32_t* pos;
  const int32_t* seq_idx;
  const int32_t* block_table;
  int B, max_pages, num_pages, page_size;
  int32_t* dev_status;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tgemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sb + OFF_BAR + 8u * (uint32_t)i; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_TSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  const int nc = a.K / 64;
  // A cluster of two takes tiles in pairs: the same 256 features for two
  // token tiles. Each CTA loads half of the weight chunk and multicasts it to
  // both, so a pair reads each weight chunk from L2 once.
  const uint32_t rank = cluster_ctarank();
  const int cl = (int)blockIdx.x >> 1, ncl = (int)gridDim.x >> 1;
  auto tile_n0 = [&](int t) { return (t / a.m_pairs) * TN; };
  auto tile_m0 = [&](int t) { return ((t % a.m_pairs) * 2 + (int)rank) * TM; };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(FULL + i), 1);
      mbar_init(bar(EMPTY + i), 2);  // both CTAs' products read the stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(TFULL + i), 1);
      mbar_init(bar(TEMPTY + i), 4);  // one arrival per epilogue warp
    }
    mbar_init(bar(FIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  cluster_sync_all();  // both CTAs' barriers initialised before any multicast

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kc = 0;
      bool ok = true;
      for (int t = cl; ok && t < a.tiles; t += ncl) {
        const int n0 = tile_n0(t), m0 = tile_m0(t);
        for (int c = 0; c < nc; ++c, ++kc) {
          const uint32_t st = kc % NST;
          ok = mbar_wait_bounded(bar(EMPTY + st), ((kc / NST) & 1) ^ 1, abort_flag, a.dev_status,
                                 WAIT_NS);
          if (!ok) break;
          const uint32_t dst = sb + st * STAGE;
          mbar_expect_tx(bar(FULL + st), STAGE);  // own X chunk + both weight halves
          tma_load_2d(dst, &tm_x, 64 * c, m0, bar(FULL + st));
          tma_load_2d_mc(dst + A_BYTES + rank * (B_BYTES / 2), &tm_w, 64 * c, n0 + (int)rank * (TN / 2),
                         bar(FULL + st), (uint16_t)3);
        }
      }
      // copies still in flight land, and the peer's products are done with
      // every stage (its commits arrive here), before the CTA may exit
      for (uint32_t k = kc > (uint32_t)NST ? kc - NST : 0; k < kc; ++k) {
        mbar_wait_drain(bar(FULL + k % NST), (k / NST) & 1, DRAIN_NS);
        mbar_wait_drain(bar(EMPTY + k % NST), (k / NST) & 1, DRAIN_NS);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      uint32_t kc = 0, i = 0;
      bool ok = true, any = false;
      for (int t = cl; ok && t < a.tiles; t += ncl, ++i) {
        const uint32_t acc = i & 1u, d = tmem + acc * TN;
        ok = mbar_wait_bounded(bar(TEMPTY + acc), ((i >> 1) & 1) ^ 1, abort_flag, a.dev_status,
                               WAIT_NS);
        if (!ok) break;
        tc_fence_after();
        for (int c = 0; c < nc; ++c, ++kc) {
          const uint32_t st = kc % NST;
          ok = mbar_wait_bounded(bar(FULL + st), (kc / NST) & 1, abort_flag, a.dev_status, WAIT_NS);
          if (!ok) break;
          tc_fence_after();
          const uint32_t xa = sb + st * STAGE, wb = xa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, sdesc_sw128(xa + kk * 32, 16, 1024), sdesc_sw128(wb + kk * 32, 16, 1024), IDESC,
                   (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit_mc(bar(EMPTY + st), (uint16_t)3);  // the stage of both CTAs
          any = true;
        }
        if (ok) mma_commit(bar(TFULL + acc));
      }
      if (!ok && any) {  // products still in flight finish before TMEM is freed
        mma_commit(bar(FIN));
        mbar_wait_drain(bar(FIN), 0, DRAIN_NS);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;         // TMEM lane quarter this warp may read
    const int r = q * 32 + lane;    // token row of the tile
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const int esz = a.out_f32 ? 4 : 2;
    uint32_t i = 0;
    for (int t = cl; t < a.tiles; t += ncl, ++i) {
      const uint32_t acc = i & 1u;
      const int n0 = tile_n0(t), m0 = tile_m0(t);
      bool waited = true;
      if (lane == 0)
        waited = mbar_wait_sleepy(bar(TFULL + acc), (i >> 1) & 1, abort_flag, a.dev_status, WAIT_NS,
                                  64);
      waited = __shfl_sync(0xffffffffu, waited, 0);
      if (!waited) break;
      mbar_try_wait(bar(TFULL + acc), (i >> 1) & 1);  // each lane acquires the completed phase
      tc_fence_after();
      // output row of this thread's token (-1: none)
      const int gm = m0 + r;
      long long row = -1;
      int ps = -1;
      if (gm < a.M) {
        if (a.epi == EPI_ROPE || a.epi == EPI_APPEND) ps = a.pos[gm];
        if (a.epi == EPI_APPEND) {
          const int sq = a.seq_idx ? a.seq_idx[gm] : gm;
          if (sq < 0 || sq >= a.B || ps < 0 || ps >= a.max_pages * a.page_size) {
            report(a.dev_status, MLA_DEV_BAD_POS);
          } else {
            const int blk = a.block_table[(size_t)sq * a.max_pages + ps / a.page_size];
            if (blk < 0 || blk >= a.num_pages) report(a.dev_status, MLA_DEV_BAD_BLOCK);
            else row = ((long long)blk * a.page_size + ps % a.page_size) * (long long)a.N;
          }
        } else {
          row = (long long)gm * a.ldo;
        }
      }
      const bool pos_ok = ps >= 0 && ps < a.max_pos;
      bool bad_pos = false;
#pragma unroll 1
      for (int b = 0; b < TN / 32; ++b) {
        uint32_t v[32];
        __syncwarp();  // rows past M skip the stores below: converge for the warp-wide load
        tmem_ld32(tmem + lane_addr + acc * TN + b * 32, v);
        tmem_ld_wait();
        if (b == TN / 32 - 1) {  // the accumulator is read out: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
        }
        const int gn0 = n0 + b * 32;
        if (row < 0 || gn0 >= a.N) continue;
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
        if (a.epi == EPI_ROPE || a.epi == EPI_APPEND) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int gn = gn0 + j;
            const int col = a.epi == EPI_ROPE ? gn % a.rope_period : gn;
            if (col < a.rope_off || col >= a.rope_off + a.d_r) continue;
            if (!pos_ok) {
              bad_pos = true;
              continue;
            }
            const float2 cs2 =
                reinterpret_cast<const float2*>(a.rope)[(size_t)ps * (a.d_r / 2) + ((col - a.rope_off) >> 1)];
            const float e = x[j], o = x[j + 1];
            x[j] = e * cs2.x - o * cs2.y;
            x[j + 1] = e * cs2.y + o * cs2.x;
          }
        }
        uint8_t* dst = reinterpret_cast<uint8_t*>(a.out) + (size_t)(row + gn0) * esz;
        if (a.vec && gn0 + 32 <= a.N) {
          if (a.out_f32) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              reinterpret_cast<float4*>(dst)[u] = make_float4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              reinterpret_cast<uint4*>(dst)[u] =
                  make_uint4(pack_bf16x2(x[8 * u], x[8 * u + 1]), pack_bf16x2(x[8 * u + 2], x[8 * u + 3]),
                             pack_bf16x2(x[8 * u + 4], x[8 * u + 5]), pack_bf16x2(x[8 * u + 6], x[8 * u + 7]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (gn0 + j >= a.N) break;
            if (a.out_f32) reinterpret_cast<float*>(dst)[j] = x[j];
            else reinterpret_cast<__nv_bfloat16*>(dst)[j] = __float2bfloat16_rn(x[j]);
          }
        }
      }
      if (bad_pos) report(a.dev_status, MLA_DEV_BAD_POS);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  cluster_sync_all();  // neither CTA leaves while the peer may still write to it
}

// [rows][cols] bf16, row stride `ld` elements, boxes of `box_rows` x 64 with
// 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                     uint32_t box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * 2) % 16 != 0)
    return cudaErrorMisalignedAddress;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult res = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tg

bool tc_tgemm_wanted(int M, int N, int K) {
  return M >= 256 && N >= 64 && K >= 64 && K % 64 == 0;
}

cudaError_t tc_tgemm_launch(const GemmArgs& g, long long ldx, cudaStream_t s) {
  using namespace tg;
  const int M = g.M, N = g.N, K = g.K;
  Args a;
  a.M = M; a.N = N; a.K = K;
  a.m_pairs = ((M + TM - 1) / TM + 1) / 2;
  a.tiles = a.m_pairs * ((N + TN - 1) / TN);
  a.epi = g.epi;
  a.out = g.out; a.ldo = g.o_ms; a.out_f32 = g.o_f32;
  a.rope = g.rope; a.max_pos = g.max_pos; a.d_r = g.d_r; a.rope_off = g.rope_off;
  a.rope_period = g.rope_period > 0 ? g.rope_period : N;
  a.pos = g.pos; a.seq_idx = g.seq_idx; a.block_table = g.block_table; a.B = g.B;
  a.max_pages = g.max_pages; a.num_pages = g.num_pages; a.page_size = g.page_size;
  a.dev_status = g.dev_status;
  {
    const long long per16 = g.o_f32 ? 4 : 8;
    const long long stride = g.epi == EPI_APPEND ? (long long)N : a.ldo;
    a.vec = (reinterpret_cast<uintptr_t>(g.out) % 16 == 0) && stride % per16 == 0;
  }
  if (g.epi != EPI_STORE && (g.rope_off % 2 != 0)) return cudaErrorInvalidValue;

  CUtensorMap tm_x, tm_w;
  cudaError_t e = make_map(&tm_x, g.a, (uint64_t)M, (uint64_t)K, (uint64_t)ldx, TM);
  if (e != cudaSuccess) return e;
  e = make_map(&tm_w, g.w, (uint64_t)N, (uint64_t)K, (uint64_t)g.w_ns, TN / 2);
  if (e != cudaSuccess) return e;
  static unsigned long long smem_done = 0;
  e = set_max_smem_once((const void*)tgemm_kernel, (int)SMEM, smem_done);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // clusters of two that can be resident at once (one CTA per SM)
  static int resident[64];
  int* res = dev >= 0 && dev < 64 ? &resident[dev] : nullptr;
  int fit = res && *res > 0 ? *res : 0;
  if (fit == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    if (cudaOccupancyMaxActiveClusters(&fit, tgemm_kernel, &cfg) != cudaSuccess || fit <= 0) {
      cudaGetLastError();
      fit = sms / 2;
    }
    if (res) *res = fit;
  }
  const int clusters = a.tiles < fit ? a.tiles : fit;
  tgemm_kernel<<<2 * clusters, THREADS, SMEM, s>>>(tm_x, tm_w, a);
  return cudaGetLastError();
}

}  // namespace mla
