// tcgen05 data-path self-test and shape/device checks for the tensor-core
// decode (DeepSeek-V2 shapes: 128 heads, d_c = 512, d_R = 64, 64-token
// pages, bf16).
//
// The self-test runs one page through tcgen05 operand layouts without
// softmax ("DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现",
// 3.2, the two products of a decode page):
//   S = Q_cat . Page^T     M = 128 heads, N = 64 tokens, K = 576: Q[:, 0:384]
//                          from TMEM, Q[:, 384:576] from SMEM, the page
//                          K-major in SMEM (TMA, 128-byte swizzle)
//   O = P . Page[:, lat]   M = 128 heads, N = 256 latent columns, K = 64
//                          tokens: P from SMEM, the page read MN-major
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

constexpr int NBAR = 3;  // operands landed, P/Q written by threads, MMAs done

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, HALF, false, true);
constexpr uint64_t WAIT_NS = 2000000000ull;

// One page, no softmax: S = Q . Page^T and O = P . Page[:, 256 r : 256 r + 256]
// through TMEM- and SMEM-sourced A operands, K-major and MN-major B operands
// with 128-byte swizzle. A diagnostic for the tensor-core data path.
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
    // warp-uniform, since the TMEM loads are warp-wide instructions
    if (__all_sync(0xffffffffu, mbar_wait_bounded(b_mma, 0, abort_flag, dev_status, WAIT_NS))) {
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
