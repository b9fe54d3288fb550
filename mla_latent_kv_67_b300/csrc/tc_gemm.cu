// tcgen05 weight-streaming GEMM for the projections of a decode step
// ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现":
// 2.1 the joint down-projection W^DKV (with W^KR of 3.2) feeding the cache,
// 2.3 the query compression W^DQ and up-projection W^UQ (with W^QR), and the
// output projection W^O of 2.2):
//
//   out[m][n] = sum_k X[m][k] W[n][k]     X [M][K] bf16 (tokens), W [N][K] bf16
//
// At decode the token count M is small (one row per sequence) and the
// weights are large, so the product is bound by reading W once. Each CTA
// takes a 128-row tile of W as the MMA's A operand (M = 128 output
// features) and a tile of up to 128 token rows as B (N = the token tile), so
// the accumulator is D[128 features][tokens] in tensor memory. A cluster of
// `cs` CTAs splits K: every CTA streams its share of the tile's K range
// through a TMA ring, then the partial accumulators are reduce-scattered
// through distributed shared memory (CTA r owns output features
// [r*128/cs, (r+1)*128/cs) of the tile and sums the cs partials in rank
// order, so results do not depend on timing). The owner applies the
// epilogue:
//   STORE   out[m * ldo + n] in fp32 or bf16;
//   ROPE    as STORE, with RoPE on the pairs (2i, 2i+1) of the columns
//           n % period >= rope_off (the decoupled query of 3.2);
//   APPEND  RoPE on n >= rope_off, then the row goes to the paged cache slot
//           of (seq_idx[m], pos[m]) (the cache row c_KV | k_R of 3.3).
//
// Warp 0 issues the TMA copies, warp 1 the MMAs (one thread each); all four
// warps run the epilogue. Every wait is bounded and reports MLA_DEV_TIMEOUT.
#include <cudaTypedefs.h>

#include "launch.h"
#include "sm100_ptx.cuh"
#include "tc_decode.h"

namespace mla {
namespace wg {

using namespace ptx;

constexpr int THREADS = 128;
constexpr int TILE_N = 128;            // output features per CTA tile (MMA M)
constexpr int MAX_MT = 128;            // token rows per CTA tile (MMA N)
constexpr uint32_t W_CHUNK = TILE_N * 128;  // one 64-wide K chunk of the W tile: 16 KB
constexpr uint32_t RING_BYTES = 96 * 1024;  // two CTAs fit on one SM
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_NS = 100000000ull;

struct Args {
  int M, N, K;
  int mt;   // token rows per tile (multiple of 16, <= MAX_MT)
  int m_tiles;  // token tiles
  int vec;      // output rows take 16-byte stores (alignment checked on the host)
  int cs;   // CTAs per cluster splitting K (1, 2, 4 or 8)
  int nst;  // ring stages
  int epi;  // Epilogue (launch.h)
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

__device__ __forceinline__ uint32_t stage_bytes(int mt) { return W_CHUNK + (uint32_t)mt * 128u; }

__global__ void __launch_bounds__(THREADS, 1)
    wgemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = a.cs, mt = a.mt, nst = a.nst;
  const uint32_t rank = cs > 1 ? cluster_ctarank() : 0u;
  // Tiles in launch order with the token tiles fastest: the CTAs in flight
  // share a few weight tiles (each read from HBM about once, the rest from
  // L2) rather than every weight tile at once. A cluster is cs consecutive
  // blocks of one row of the grid, so all its CTAs get the same tile.
  const int tile = (int)((blockIdx.y * gridDim.x + blockIdx.x) / (unsigned)cs);
  const int n0 = (tile / a.m_tiles) * TILE_N;
  const int m0 = (tile % a.m_tiles) * mt;
  const int nc = a.K / 64;
  const int c0 = (int)(rank * nc / cs), c1 = (int)((rank + 1) * nc / cs);
  const uint32_t SB = stage_bytes(mt);
  // barriers after the ring: full[nst], empty[nst], done; then the TMEM
  // address slot and the abort flag
  const uint32_t bar0 = sb + (uint32_t)nst * SB;
  auto full = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty = [&](int i) { return bar0 + 8u * (uint32_t)(nst + i); };
  const uint32_t done = bar0 + 8u * (uint32_t)(2 * nst);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + (size_t)nst * SB + 8 * (2 * nst + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const uint32_t tcols = mt <= 32 ? 32u : (mt <= 64 ? 64u : 128u);

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    for (int i = 0; i < nst; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tslot), tcols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    for (int c = c0; c < c1; ++c, ++issued) {
      const int i = c - c0, st = i % nst;
      if (!mbar_wait_bounded(empty(st), ((i / nst) & 1) ^ 1, abort_flag, a.dev_status, WAIT_NS))
        break;
      const uint32_t dst = sb + (uint32_t)st * SB;
      mbar_expect_tx(full(st), SB);
      tma_load_2d(dst, &tm_w, 64 * c, n0, full(st));
      tma_load_2d(dst + W_CHUNK, &tm_x, 64 * c, m0, full(st));
    }
    // copies still in flight land before the CTA may exit
    for (int i = issued > nst ? issued - nst : 0; i < issued; ++i)
      mbar_wait_drain(full(i % nst), (i / nst) & 1, DRAIN_NS);
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issue
    const uint32_t idesc = idesc_bf16_f32(TILE_N, mt, false, false);
    bool ok = true, any = false;
    for (int c = c0; c < c1; ++c) {
      const int i = c - c0, st = i % nst;
      ok = mbar_wait_bounded(full(st), (i / nst) & 1, abort_flag, a.dev_status, WAIT_NS);
      if (!ok) break;
      tc_fence_after();
      const uint32_t wt = sb + (uint32_t)st * SB, xt = wt + W_CHUNK;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(tmem, sdesc_sw128(wt + kk * 32, 16, 1024), sdesc_sw128(xt + kk * 32, 16, 1024), idesc,
               (c > c0 || kk > 0) ? 1u : 0u);
      mma_commit(empty(st));
      if (c == c1 - 1) mma_commit(done);  // back to back with the last products in flight
      any = true;
    }
    if (!ok || !any) {
      // the epilogue must not wait forever: drain what was issued, then arrive
      if (any) {
        mma_commit(done);
        mbar_wait_drain(done, 0, DRAIN_NS);
      } else {
        mbar_arrive(done);
      }
    }
  }
  __syncwarp();

  // ---------------------------------------------------------- epilogue
  // 1. every CTA's partial accumulator is complete and its ring is idle
  // one lane per warp polls, sleeping between polls, so the waiting warps
  // take no issue slots from the producer and the MMA issuer
  bool waited = true;
  if (lane == 0) waited = mbar_wait_sleepy(done, 0, abort_flag, a.dev_status, WAIT_NS, 64);
  waited = __shfl_sync(0xffffffffu, waited, 0);
  if (waited) mbar_try_wait(done, 0);  // each lane acquires the completed phase
  const bool mma_ok = __all_sync(0xffffffffu, waited && !*abort_flag);
  tc_fence_after();
  if (cs == 1) {
    // The whole K range is in this CTA's accumulator: thread r (TMEM lane r)
    // holds output feature n0 + r for every token of the tile. It reads 16
    // tokens at a time from TMEM, applies RoPE (the pair partner is the
    // neighbouring lane) and parks the values in a [tokens][128 features]
    // tile in the idle ring; then the CTA writes every token's 128 features
    // as one contiguous run with 16-byte stores. (Without the alignment for
    // 16-byte stores each warp stores its 32 features of a token directly.)
    const int r = threadIdx.x, gn = n0 + r;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    const int esz = a.out_f32 ? 4 : 2;
    const int RB = TILE_N * esz;  // bytes of one staged token row
    uint8_t* stg = smem;          // [mt][TILE_N] values, reuses the ring
    long long* rowoff = reinterpret_cast<long long*>(smem + (size_t)mt * RB);  // [mt] output row (elements), -1: none
    int rk = -1;  // RoPE pair of this feature (-1: none) and its side
    bool odd = false;
    if (a.epi == EPI_ROPE || a.epi == EPI_APPEND) {
      const int col = a.epi == EPI_ROPE ? gn % a.rope_period : gn;
      if (col >= a.rope_off && col < a.rope_off + a.d_r) {
        rk = (col - a.rope_off) >> 1;
        odd = ((col - a.rope_off) & 1) != 0;
      }
    }
    // the output row of token r of the tile (one thread per token)
    long long my_row = -1;
    if (r < mt && m0 + r < a.M && mma_ok) {
      const int gm = m0 + r;
      if (a.epi == EPI_APPEND) {
        const int sq = a.seq_idx ? a.seq_idx[gm] : gm;
        const int ps = a.pos[gm];
        if (sq < 0 || sq >= a.B || ps < 0 || ps >= a.max_pages * a.page_size) {
          report(a.dev_status, MLA_DEV_BAD_POS);
        } else {
          const int blk = a.block_table[(size_t)sq * a.max_pages + ps / a.page_size];
          if (blk < 0 || blk >= a.num_pages) report(a.dev_status, MLA_DEV_BAD_BLOCK);
          else my_row = ((long long)blk * a.page_size + ps % a.page_size) * (long long)a.N;
        }
      } else {
        my_row = (long long)gm * a.ldo;
      }
    }
    if (a.vec && r < mt) rowoff[r] = my_row;
    for (int j0 = 0; j0 < mt; j0 += 16) {
      uint32_t v[16];
      if (mma_ok) {
        tmem_ld16(taddr + j0, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = 0u;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int j = j0 + u, gm = m0 + j;
        float x = __uint_as_float(v[u]);
        const float partner = __shfl_xor_sync(0xffffffffu, x, 1);
        if (gm >= a.M || !mma_ok) continue;
        if (rk >= 0) {
          const int ps = a.pos[gm];
          if (ps < 0 || ps >= a.max_pos) {
            report(a.dev_status, MLA_DEV_BAD_POS);
          } else {
            const float2 cs2 = reinterpret_cast<const float2*>(a.rope)[(size_t)ps * (a.d_r / 2) + rk];
            x = odd ? partner * cs2.y + x * cs2.x : x * cs2.x - partner * cs2.y;
          }
        }
        if (a.vec) {
          if (a.out_f32) reinterpret_cast<float*>(stg + (size_t)j * RB)[r] = x;
          else reinterpret_cast<__nv_bfloat16*>(stg + (size_t)j * RB)[r] = __float2bfloat16_rn(x);
          continue;
        }
        if (gn >= a.N) continue;
        long long o;
        if (a.epi == EPI_APPEND) {
          const int sq = a.seq_idx ? a.seq_idx[gm] : gm;
          const int ps = a.pos[gm];
          if (sq < 0 || sq >= a.B || ps < 0 || ps >= a.max_pages * a.page_size) continue;
          const int blk = a.block_table[(size_t)sq * a.max_pages + ps / a.page_size];
          if (blk < 0 || blk >= a.num_pages) continue;
          o = ((long long)blk * a.page_size + ps % a.page_size) * (long long)a.N + gn;
        } else {
          o = (long long)gm * a.ldo + gn;
        }
        if (a.out_f32) reinterpret_cast<float*>(a.out)[o] = x;
        else reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(x);
      }
    }
    if (a.vec) {
      __syncthreads();
      const int per16 = 16 / esz;        // elements per 16-byte piece
      const int cpr = RB / 16;           // pieces per token row
      for (int c = r; c < mt * cpr; c += THREADS) {
        const int j = c / cpr, q = c % cpr;
        const long long row = rowoff[j];
        const int g0 = n0 + q * per16;
        if (row < 0 || g0 >= a.N) continue;
        const uint4 val = *reinterpret_cast<const uint4*>(stg + (size_t)j * RB + (size_t)q * 16);
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.out) + (size_t)(row + g0) * esz) = val;
      }
    }
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, tcols);
    }
    return;
  }
  const int R = TILE_N / cs;  // output features each CTA of the cluster owns
  float* red = reinterpret_cast<float*>(smem);  // [cs][mt][R], reuses the ring
  if (cs > 1) cluster_sync_all();
  else __syncthreads();
  // 2. row r of this CTA's partial (thread = TMEM lane = feature) goes to
  //    its owner's buffer, slot [rank][m][r % R]
  {
    const int r = threadIdx.x;
    const uint32_t owner = (uint32_t)(r / R);
    const uint32_t base = mapa_shared(smem_u32(red) + 4u * (uint32_t)((rank * mt) * R + (r % R)), owner);
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    for (int j = 0; j < mt; j += 16) {
      uint32_t v[16];
      if (mma_ok) {
        tmem_ld16(taddr + j, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = 0u;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) st_cluster_u32(base + 4u * (uint32_t)((j + u) * R), v[u]);
    }
  }
  tc_fence_before();
  if (cs > 1) cluster_sync_all();
  else __syncthreads();
  // 3. the owner sums the partials in rank order and applies the epilogue;
  //    consecutive threads take consecutive features, so a RoPE pair sits in
  //    lanes (2i, 2i+1) and every store of a warp is contiguous
  const int per = mt * R;  // a multiple of 128 (mt >= 16, cs <= 8)
  for (int idx = threadIdx.x; idx < per; idx += THREADS) {
    const int m = idx / R, r = idx % R;
    float v = 0.f;
    for (int s = 0; s < cs; ++s) v += red[(s * mt + m) * R + r];
    const int gm = m0 + m, gn = n0 + (int)rank * R + r;
    const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
    if (gm >= a.M || gn >= a.N || !mma_ok) continue;
    if (a.epi == EPI_ROPE || a.epi == EPI_APPEND) {
      const int col = a.epi == EPI_ROPE ? gn % a.rope_period : gn;
      if (col >= a.rope_off && col < a.rope_off + a.d_r) {
        const int ps = a.pos[gm];
        if (ps < 0 || ps >= a.max_pos) {
          report(a.dev_status, MLA_DEV_BAD_POS);
        } else {
          const int k = (col - a.rope_off) >> 1;
          const float2 cs2 = reinterpret_cast<const float2*>(a.rope)[(size_t)ps * (a.d_r / 2) + k];
          v = ((col - a.rope_off) & 1) == 0 ? v * cs2.x - partner * cs2.y
                                            : partner * cs2.y + v * cs2.x;
        }
      }
    }
    size_t o;
    if (a.epi == EPI_APPEND) {
      const int sq = a.seq_idx ? a.seq_idx[gm] : gm;
      const int ps = a.pos[gm];
      if (sq < 0 || sq >= a.B || ps < 0 || ps >= a.max_pages * a.page_size) {
        report(a.dev_status, MLA_DEV_BAD_POS);
        continue;
      }
      const int blk = a.block_table[(size_t)sq * a.max_pages + ps / a.page_size];
      if (blk < 0 || blk >= a.num_pages) {
        report(a.dev_status, MLA_DEV_BAD_BLOCK);
        continue;
      }
      o = ((size_t)blk * a.page_size + ps % a.page_size) * (size_t)a.N + gn;
    } else {
      o = (size_t)gm * (size_t)a.ldo + gn;
    }
    if (a.out_f32) reinterpret_cast<float*>(a.out)[o] = v;
    else reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(v);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
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

// [rows][cols] bf16, row stride `ld` elements, boxes of `box_rows` x 64
// with 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                     uint32_t box_rows) {
  auto fn = encode_fn();
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

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return sms;
}

}  // namespace wg

bool tc_gemm_supported(int M, int N, int K, long long ldx) {
  return M > 0 && N > 0 && K >= 64 && K % 64 == 0 && ldx % 8 == 0 && tc_decode_supported(128, 512, 64, 64);
}

cudaError_t tc_gemm_launch(const GemmArgs& g, long long ldx, cudaStream_t s) {
  using namespace wg;
  const int M = g.M, N = g.N, K = g.K;
  const int mt_full = M < MAX_MT ? M : MAX_MT;
  const int mt = (mt_full + 15) / 16 * 16;
  const int n_tiles = (N + TILE_N - 1) / TILE_N, m_tiles = (M + mt - 1) / mt;
  const int nc = K / 64;
  // split K over a cluster until the grid covers every SM (two CTAs fit on
  // one SM), without more CTAs than K chunks
  const int sms = device_sms();
  int cs = 1;
  while (cs < 8 && 2 * cs <= nc && n_tiles * m_tiles * cs * 2 <= 2 * sms &&
         n_tiles * m_tiles * cs < sms)
    cs *= 2;
  Args a;
  a.M = M; a.N = N; a.K = K; a.mt = mt; a.cs = cs; a.m_tiles = m_tiles;
  const uint32_t SB = W_CHUNK + (uint32_t)mt * 128u;
  a.nst = (int)(RING_BYTES / SB);
  if (a.nst > 8) a.nst = 8;
  a.epi = g.epi;
  a.out = g.out; a.ldo = g.o_ms; a.out_f32 = g.o_f32;
  a.rope = g.rope; a.max_pos = g.max_pos; a.d_r = g.d_r; a.rope_off = g.rope_off;
  a.rope_period = g.rope_period > 0 ? g.rope_period : N;
  a.pos = g.pos; a.seq_idx = g.seq_idx; a.block_table = g.block_table; a.B = g.B;
  a.max_pages = g.max_pages; a.num_pages = g.num_pages; a.page_size = g.page_size;
  a.dev_status = g.dev_status;
  {
    // 16-byte output stores need every 8 (bf16) or 4 (fp32) features of a
    // row in one aligned piece: an aligned base, the row stride and N in
    // whole pieces
    const long long per16 = g.o_f32 ? 4 : 8;
    const long long stride = g.epi == EPI_APPEND ? (long long)N : a.ldo;
    a.vec = (reinterpret_cast<uintptr_t>(g.out) % 16 == 0) && stride % per16 == 0 && N % per16 == 0;
  }
  if (g.epi != EPI_STORE && (g.rope_off % 2 != 0)) return cudaErrorInvalidValue;

  CUtensorMap tm_w, tm_x;
  cudaError_t e = make_map(&tm_w, g.w, (uint64_t)N, (uint64_t)K, (uint64_t)g.w_ns, TILE_N);
  if (e != cudaSuccess) return e;
  e = make_map(&tm_x, g.a, (uint64_t)M, (uint64_t)K, (uint64_t)ldx, (uint32_t)mt);
  if (e != cudaSuccess) return e;

  const uint32_t smem = (uint32_t)a.nst * SB + 8u * (2u * a.nst + 1u) + 16u + 1024u;
  static unsigned long long smem_done = 0;
  e = set_max_smem_once((const void*)wgemm_kernel, (int)(RING_BYTES + 8 * 17 + 16 + 1024), smem_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_tiles * cs), (unsigned)m_tiles);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wgemm_kernel, tm_w, tm_x, a);
}

}  // namespace mla
