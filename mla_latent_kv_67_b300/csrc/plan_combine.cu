// Split planner (a4) and split-KV combine (a6).
//
// The planner turns seq_lens into a WorkerPlan per worker and a SeqPlan per
// sequence (layout in common.cuh); it runs on the device so a decode step
// needs no host round trip and can be captured in a CUDA graph.
#include <math.h>

#include "common.cuh"
#include "launch.h"

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

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ seq_lens, int B,
                                                    int max_pages, int page_size, int workers,
                                                    int path, char* ws, WorkspaceLayout L,
                                                    int32_t* dev_status) {
  __shared__ int warp_sums[32];
  __shared__ int carry_s;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws + L.header);
  SeqPlan* seqs = reinterpret_cast<SeqPlan*>(ws + L.seqs);
  WorkerPlan* wk = reinterpret_cast<WorkerPlan*>(ws + L.workers);

  // pass 1: validated page counts and their exclusive prefix sum
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int pages = 0, len = 0;
    if (b < B) {
      len = seq_lens[b];
      if (len < 1 || (long long)len > (long long)max_pages * page_size) {
        report(dev_status, MLA_DEV_BAD_LEN);
        len = 0;
      }
      pages = (len + page_size - 1) / page_size;
    }
    const int incl = block_inclusive_scan(pages, warp_sums);
    const int carry = carry_s;
    if (b < B) {
      seqs[b].page_begin = carry + incl - pages;
      seqs[b].pages = pages;
      seqs[b].len = len;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry_s = carry + incl;
    __syncthreads();
  }
  const int total = carry_s;
  const int per = total > 0 ? (total + workers - 1) / workers : 1;

  // pass 2: which workers touch each sequence, and its partial slots
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int slots = 0;
    if (b < B) {
      const int pb = seqs[b].page_begin, np = seqs[b].pages;
      int first = 0, n = 0;
      if (np > 0) {
        first = pb / per;
        n = (pb + np - 1) / per - first + 1;
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

  // pass 3: each worker's (sequence, page) range, by binary search on
  // page_begin (the last sequence whose first global page is <= x; a
  // sequence with no pages shares its begin with the next one, so the
  // search lands on a sequence that owns page x).
  for (int g = threadIdx.x; g < workers; g += blockDim.x) {
    WorkerPlan w;
    const int x0 = g * per;
    const int x1 = min(x0 + per, total) - 1;  // inclusive
    w.n_pages = x1 >= x0 ? x1 - x0 + 1 : 0;
    w.seq_begin = w.page_begin = w.seq_end = w.page_end = 0;
    w.pad[0] = w.pad[1] = w.pad[2] = 0;
    if (w.n_pages > 0) {
      int xs[2] = {x0, x1};
      for (int e = 0; e < 2; ++e) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (seqs[mid].page_begin <= xs[e]) lo = mid; else hi = mid - 1;
        }
        if (e == 0) { w.seq_begin = lo; w.page_begin = xs[e] - seqs[lo].page_begin; }
        else        { w.seq_end = lo;   w.page_end = xs[e] - seqs[lo].page_begin; }
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
  }
}

// One block per (sequence, head): merge the sequence's partial slots.
__global__ void __launch_bounds__(128) combine_kernel(const char* __restrict__ ws, WorkspaceLayout L,
                                                      int n_h, int d_c, float* __restrict__ o_lat,
                                                      float* __restrict__ lse) {
  const int b = blockIdx.x, h = blockIdx.y;
  const SeqPlan sp = reinterpret_cast<const SeqPlan*>(ws + L.seqs)[b];
  float* o = o_lat + ((size_t)b * n_h + h) * d_c;
  if (sp.n_splits == 1) return;  // written by the decode kernel
  if (sp.n_splits == 0) {        // invalid length: defined, empty result
    for (int c = threadIdx.x; c < d_c; c += blockDim.x) o[c] = 0.f;
    if (threadIdx.x == 0) lse[(size_t)b * n_h + h] = -INFINITY;
    return;
  }
  const float* lp = reinterpret_cast<const float*>(ws + L.lse_part);
  const float* op = reinterpret_cast<const float*>(ws + L.o_part);
  float m = -INFINITY;
  for (int s = 0; s < sp.n_splits; ++s) m = fmaxf(m, lp[(size_t)(sp.slot_begin + s) * n_h + h]);
  float z = 0.f;
  for (int s = 0; s < sp.n_splits; ++s) {
    const float l = lp[(size_t)(sp.slot_begin + s) * n_h + h];
    z += l == -INFINITY ? 0.f : expf(l - m);
  }
  const float inv = 1.f / z;
  for (int c = threadIdx.x; c < d_c; c += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < sp.n_splits; ++s) {
      const size_t slot = (size_t)(sp.slot_begin + s);
      const float l = lp[slot * n_h + h];
      if (l == -INFINITY) continue;
      acc += expf(l - m) * op[(slot * n_h + h) * d_c + c];
    }
    o[c] = acc * inv;
  }
  if (threadIdx.x == 0) lse[(size_t)b * n_h + h] = m + logf(z);
}

cudaError_t launch_plan(const int32_t* seq_lens, int B, int max_pages, int page_size, int workers,
                        int path, void* ws, const WorkspaceLayout& L, int32_t* dev_status,
                        cudaStream_t s) {
  plan_kernel<<<1, 1024, 0, s>>>(seq_lens, B, max_pages, page_size, workers, path, (char*)ws, L,
                                 dev_status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* ws, const WorkspaceLayout& L, int B, int n_h, int d_c,
                           float* o_lat, float* lse, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  combine_kernel<<<dim3(B, n_h), 128, 0, s>>>((const char*)ws, L, n_h, d_c, o_lat, lse);
  return cudaGetLastError();
}

}  // namespace mla
