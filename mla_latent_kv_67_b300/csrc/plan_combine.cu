// Split planner (a4) and split-KV combine (a6).
//
// The planner turns seq_lens into a WorkerPlan per worker and a SeqPlan per
// sequence (layout in common.cuh); it runs on the device so a decode step
// needs no host round trip and can be captured in a CUDA graph.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "sm100_ptx.cuh"

namespace mla {

// Block-wide inclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_inclusive_scan(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int s = lane < nw ? warp_sums[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += t;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  if (warp > 0) v += warp_sums[warp - 1];
  __syncthreads();
  return v;
}

constexpr int PLAN_SMEM_SEQS = 4096;  // sequences whose cost prefix stays in shared memory

// Work split. Every worker pays a fixed cost for each sequence it touches
// (bringing the sequence's Q in, writing its partial O out) on top of one
// unit per page. Each sequence with pages therefore gets `c_seg` cost units
// in front of its pages, the cost axis is cut into `workers` equal ranges,
// and worker g takes the pages whose units fall in its range: a worker that
// starts a sequence inside its range gets c_seg pages fewer.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ seq_lens, int B,
                                                    int q_len, int max_pages, int page_size,
                                                    int workers,
                                                    int path, int part_bf16, int c_seg, char* ws,
                                                    WorkspaceLayout L, int32_t* dev_status) {
  __shared__ int warp_sums[32];
  __shared__ int carry_s, ccarry_s;
  __shared__ int vend_s[PLAN_SMEM_SEQS], pages_s[PLAN_SMEM_SEQS];
  const bool in_smem = B <= PLAN_SMEM_SEQS;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws + L.header);
  SeqPlan* seqs = reinterpret_cast<SeqPlan*>(ws + L.seqs);
  WorkerPlan* wk = reinterpret_cast<WorkerPlan*>(ws + L.workers);

  // pass 1: validated page counts, their exclusive prefix sum, and the
  // prefix sum of cost units (pages + c_seg per sequence with pages)
  if (threadIdx.x == 0) carry_s = ccarry_s = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int pages = 0, len = 0;
    if (b < B) {
      // query row b is new token b % q_len of sequence b / q_len
      len = seq_lens[b / q_len] - (q_len - 1 - b % q_len);
      if (len < 1 || (long long)len > (long long)max_pages * page_size) {
        report(dev_status, MLA_DEV_BAD_LEN);
        len = 0;
      }
      pages = (len + page_size - 1) / page_size;
    }
    const int units = pages > 0 ? pages + c_seg : 0;
    const int incl = block_inclusive_scan(pages, warp_sums);
    const int cincl = block_inclusive_scan(units, warp_sums);
    const int carry = carry_s, ccarry = ccarry_s;
    if (b < B) {
      seqs[b].page_begin = carry + incl - pages;
      seqs[b].cost_begin = ccarry + cincl - units;
      seqs[b].pages = pages;
      seqs[b].len = len;
      if (in_smem) {
        vend_s[b] = ccarry + cincl;
        pages_s[b] = pages;
      }
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      carry_s = carry + incl;
      ccarry_s = ccarry + cincl;
    }
    __syncthreads();
  }
  const int total = carry_s, total_units = ccarry_s;
  const int per = total_units > 0 ? (total_units + workers - 1) / workers : 1;
  auto vend = [&](int b) { return in_smem ? vend_s[b] : seqs[b].cost_begin + (seqs[b].pages > 0 ? seqs[b].pages + c_seg : 0); };
  auto npages = [&](int b) { return in_smem ? pages_s[b] : seqs[b].pages; };

  // pass 2: which workers touch each sequence, and its partial slots
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int slots = 0;
    if (b < B) {
      const int np = npages(b);
      int first = 0, n = 0;
      if (np > 0) {
        const int rs = vend(b) - np;  // cost unit of the first page
        first = rs / per;
        n = (rs + np - 1) / per - first + 1;
      }
      seqs[b].first_worker = first;
      seqs[b].n_splits = n;
      slots = n > 1 ? n : 0;
    }
    const int incl = block_inclusive_scan(slots, warp_sums);
    const int carry = carry_s;
    if (b < B) seqs[b].slot_begin = carry + incl - slots;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry_s = carry + incl;
    __syncthreads();
  }
  const int num_slots = carry_s;

  // pass 3: each worker's (sequence, page) range. Its units are [x0, x1];
  // the first page is in the first sequence whose units end after x0 (it
  // has pages: a sequence without pages ends where its predecessor does),
  // the last in the last sequence with pages whose first page's unit is
  // <= x1.
  auto first_end_after = [&](int x) {  // smallest b with vend(b) > x, or B
    int lo = 0, hi = B;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (vend(mid) > x) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  for (int g = threadIdx.x; g < workers; g += blockDim.x) {
    WorkerPlan w;
    w.seq_begin = w.page_begin = w.seq_end = w.page_end = w.n_pages = 0;
    w.pad[0] = w.pad[1] = w.pad[2] = 0;
    const int x0 = g * per;
    const int x1 = min(x0 + per, total_units) - 1;  // inclusive
    if (x1 >= x0) {
      const int bf = first_end_after(x0);
      const int rsf = vend(bf) - npages(bf);
      const int pf = max(0, x0 - rsf);
      if (rsf + pf <= x1) {  // the range holds at least one page
        int bl = first_end_after(x1);  // < B: the last sequence ends at total_units > x1
        int pl;
        const int rsl = vend(bl) - npages(bl);
        if (rsl <= x1) {
          pl = x1 - rsl;
        } else {  // x1 falls in bl's leading units: the last page before them
          bl -= 1;
          while (bl > bf && npages(bl) == 0) --bl;
          pl = npages(bl) - 1;
        }
        w.seq_begin = bf;
        w.page_begin = pf;
        w.seq_end = bl;
        w.page_end = pl;
        w.n_pages = (seqs[bl].page_begin + pl) - (seqs[bf].page_begin + pf) + 1;
      }
    }
    wk[g] = w;
  }
  if (threadIdx.x == 0) {
    hdr->workers = workers;
    hdr->per_worker = per;
    hdr->total_pages = total;
    hdr->num_slots = num_slots;
    hdr->batch = B;
    hdr->path = path;
    hdr->part_bf16 = part_bf16;
  }
}

// One warp per (sequence, head), four heads per block: merge the sequence's
// partial slots, o = sum_s exp(lse_s - lse) o_s with lse = log sum_s
// exp(lse_s). Each lane owns float4 columns lane, lane + 32, ... so every
// load and store of the warp is one contiguous row piece. P16: the partial
// slots hold bf16 (else fp32).
template <bool P16>
__device__ __forceinline__ void merge_row(const char* __restrict__ ws, const WorkspaceLayout& L,
                                          const SeqPlan& sp, int b, int h, int lane, int n_h,
                                          int d_c, float* __restrict__ o_lat,
                                          float* __restrict__ lse) {
  float4* o = reinterpret_cast<float4*>(o_lat + ((size_t)b * n_h + h) * d_c);
  const int n4 = d_c / 4;
  const float* lp = reinterpret_cast<const float*>(ws + L.lse_part);
  const int n = sp.n_splits;
  constexpr int MAXV = 4;  // float4 columns per lane held in registers (d_c <= 512)
  constexpr int RS = 4;    // splits whose rows are loaded per round
  // One round: the rows of splits s0 .. s0 + RS - 1 (a split past the end
  // re-reads the last one and gets weight 0), all loads issued together.
  float4 x[RS][MAXV];
  auto load_round = [&](int s0) {
#pragma unroll
    for (int t = 0; t < RS; ++t) {
      const size_t slot = (size_t)(sp.slot_begin + min(s0 + t, n - 1));
      const size_t e0 = (slot * n_h + h) * d_c;
#pragma unroll
      for (int v = 0; v < MAXV; ++v) {
        const int i = lane + 32 * v;
        if (i >= n4)
          x[t][v] = make_float4(0.f, 0.f, 0.f, 0.f);
        else if (P16)
          x[t][v] = load_part_bf16x4(ws + L.o_part, e0 + 4 * (size_t)i);
        else
          x[t][v] = ptx::ld_nc_v4(
              reinterpret_cast<const float4*>(reinterpret_cast<const float*>(ws + L.o_part) + e0) + i);
      }
    }
  };
  // the first round's rows and the splits' lse values in flight together
  load_round(0);
  const float l_lane = lane < n ? lp[(size_t)(sp.slot_begin + lane) * n_h + h] : -INFINITY;
  float m = l_lane;
  for (int s0 = 32; s0 < n; s0 += 32)  // more than 32 splits: rare
    if (s0 + lane < n) m = fmaxf(m, lp[(size_t)(sp.slot_begin + s0 + lane) * n_h + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = l_lane == -INFINITY ? 0.f : expf(l_lane - m);
  for (int s0 = 32; s0 < n; s0 += 32)
    if (s0 + lane < n) {
      const float l = lp[(size_t)(sp.slot_begin + s0 + lane) * n_h + h];
      z += l == -INFINITY ? 0.f : expf(l - m);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float inv = 1.f / z;
  float4 acc[MAXV];
#pragma unroll
  for (int v = 0; v < MAXV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n; s0 += RS) {
    if (s0 > 0) load_round(s0);
#pragma unroll
    for (int t = 0; t < RS; ++t) {
      const int sidx = s0 + t;
      float l = __shfl_sync(0xffffffffu, l_lane, sidx & 31);
      if (sidx >= 32 && sidx < n) l = lp[(size_t)(sp.slot_begin + sidx) * n_h + h];
      const float wgt = (sidx < n && l != -INFINITY) ? expf(l - m) * inv : 0.f;
#pragma unroll
      for (int v = 0; v < MAXV; ++v) {
        acc[v].x = fmaf(wgt, x[t][v].x, acc[v].x);
        acc[v].y = fmaf(wgt, x[t][v].y, acc[v].y);
        acc[v].z = fmaf(wgt, x[t][v].z, acc[v].z);
        acc[v].w = fmaf(wgt, x[t][v].w, acc[v].w);
      }
    }
  }
#pragma unroll
  for (int v = 0; v < MAXV; ++v) {
    const int i = lane + 32 * v;
    if (i < n4) o[i] = acc[v];
  }
  if (lane == 0) lse[(size_t)b * n_h + h] = m + logf(z);
}


__global__ void __launch_bounds__(128) combine_kernel(const char* __restrict__ ws, WorkspaceLayout L,
                                                      int n_h, int d_c, float* __restrict__ o_lat,
                                                      float* __restrict__ lse) {
  const int b = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (h >= n_h) return;
  const SeqPlan sp = reinterpret_cast<const SeqPlan*>(ws + L.seqs)[b];
  const bool p16 = reinterpret_cast<const PlanHeader*>(ws + L.header)->part_bf16 != 0;
  if (sp.n_splits == 1) return;  // written by the decode kernel
  if (sp.n_splits == 0) {        // invalid length: defined, empty result
    float4* o = reinterpret_cast<float4*>(o_lat + ((size_t)b * n_h + h) * d_c);
    for (int i = lane; i < d_c / 4; i += 32) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) lse[(size_t)b * n_h + h] = -INFINITY;
    return;
  }
  if (p16) merge_row<true>(ws, L, sp, b, h, lane, n_h, d_c, o_lat, lse);
  else merge_row<false>(ws, L, sp, b, h, lane, n_h, d_c, o_lat, lse);
}

cudaError_t launch_plan(const int32_t* seq_lens, int B, int q_len, int max_pages, int page_size,
                        int workers, int path, bool part_bf16, void* ws, const WorkspaceLayout& L,
                        int32_t* dev_status, cudaStream_t s) {
  // the tcgen05 kernel's per-sequence cost (Q fetch, O write-out) is worth
  // about four pages; the SIMT kernel's is small next to its page cost
  const int c_seg = path >= 1 ? 4 : 0;
  plan_kernel<<<1, 1024, 0, s>>>(seq_lens, B * q_len, q_len, max_pages, page_size, workers, path,
                                 part_bf16 ? 1 : 0, c_seg, (char*)ws, L, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* ws, const WorkspaceLayout& L, int B, int n_h, int d_c,
                           float* o_lat, float* lse, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  combine_kernel<<<dim3(B, (n_h + 3) / 4), 128, 0, s>>>((const char*)ws, L, n_h, d_c, o_lat, lse);
  return cudaGetLastError();
}

}  // namespace mla
