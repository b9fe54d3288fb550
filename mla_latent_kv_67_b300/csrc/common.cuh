// Shared device helpers and the decode workspace layout.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mla_b300.h"

namespace mla {

// ------------------------------------------------------------ element I/O
__device__ __forceinline__ float load_elem(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// Four consecutive bf16 partial elements starting at element e (e a
// multiple of 4) of a bf16 array at byte address base, as floats.
__device__ __forceinline__ float4 load_part_bf16x4(const char* base, size_t e) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(base) + e / 4);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ void report(int32_t* dev_status, int bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

// ------------------------------------------------------- plan / workspace
// The decode plan cuts the concatenation of all sequences' pages into
// `workers` contiguous ranges of `per_worker` pages. Worker g owns global
// pages [g*per, min((g+1)*per, total)). A sequence touched by k > 1 workers
// owns k partial slots starting at `slot_begin`; its k-th worker (in order)
// writes slot slot_begin + k. A slot is the normalised partial output
// [n_h][d_c] (element ((slot * n_h + h) * d_c + c) of the o_part region, in
// bf16 when the header's part_bf16 is set, else fp32) and its lse [n_h]
// (fp32).
struct PlanHeader {
  int32_t workers;      // number of workers the plan was made for
  int32_t per_worker;   // cost units per worker (>= 1)
  int32_t total_pages;  // sum over sequences
  int32_t num_slots;    // partial slots used
  int32_t batch;
  int32_t path;         // decode kernel the plan is for (0 SIMT, 1 and 2 tcgen05)
  int32_t part_bf16;    // partial slots hold bf16 (bf16 / FP8 caches) or fp32 (fp32 cache)
  int32_t pad;
};

struct SeqPlan {
  int32_t page_begin;   // first global page of the sequence
  int32_t pages;        // pages of the sequence
  int32_t first_worker; // worker holding its first page
  int32_t n_splits;     // workers touching it
  int32_t slot_begin;   // first partial slot (valid if n_splits > 1)
  int32_t len;          // tokens (validated copy of seq_lens[b])
  int32_t cost_begin;   // first cost unit (see plan_kernel)
  int32_t pad;
};

struct WorkerPlan {
  int32_t seq_begin, page_begin;  // first (sequence, page-in-sequence)
  int32_t seq_end, page_end;      // last  (sequence, page-in-sequence), inclusive
  int32_t n_pages;                // 0 = idle worker
  int32_t pad[3];
};

struct WorkspaceLayout {
  size_t header, seqs, workers, o_part, lse_part, total;
  int max_slots;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// max_slots: every interior cut adds one slot to one sequence and a split
// sequence has one more slot than cuts, so slots <= 2 * (workers - 1) + 1.
__host__ __device__ inline WorkspaceLayout workspace_layout(int B, int workers, int n_h, int d_c) {
  WorkspaceLayout L;
  L.max_slots = 2 * workers;
  size_t off = 0;
  L.header = off;   off = align_up(off + sizeof(PlanHeader), 256);
  L.seqs = off;     off = align_up(off + sizeof(SeqPlan) * (size_t)(B > 0 ? B : 1), 256);
  L.workers = off;  off = align_up(off + sizeof(WorkerPlan) * (size_t)workers, 256);
  L.o_part = off;   off = align_up(off + sizeof(float) * (size_t)L.max_slots * n_h * d_c, 256);
  L.lse_part = off; off = align_up(off + sizeof(float) * (size_t)L.max_slots * n_h, 256);
  L.total = off;
  return L;
}

}  // namespace mla
