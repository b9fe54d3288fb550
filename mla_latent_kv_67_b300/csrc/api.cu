// C ABI entry points: argument checks on the host, then kernel dispatch.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <string>

#include "common.cuh"
#include "launch.h"
#include "tc_decode.h"

using namespace mla;

namespace {

thread_local std::string g_last_error;
int g_forced_path = -1;

mla_status fail(mla_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = std::string(mla_status_string(st)) + ": " + buf;
  return st;
}

mla_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MLA_OK;
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define REQUIRE(cond, ...) \
  do {                     \
    if (!(cond)) return fail(MLA_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// A projection: for bf16 operands of a shape they take, the tcgen05 tile
// GEMM when there are many tokens (the product is then tensor-core bound)
// and the weight-streaming GEMM otherwise (few tokens: bound by reading the
// weights); the CUDA-core GEMM for the rest (fp32, odd K, or the SIMT path
// forced for cross-checks).
cudaError_t projection(const GemmArgs& g, cudaStream_t s) {
  if (!g.a_f32 && !g.w_f32 && g.G == 1 && g.w_ks == 1 && g_forced_path != 0 &&
      aligned16(g.a) && aligned16(g.w) && g.w_ns % 8 == 0 &&
      tc_gemm_supported(g.M, g.N, g.K, g.a_ms))
    return tc_tgemm_wanted(g.M, g.N, g.K) ? tc_tgemm_launch(g, g.a_ms, s)
                                           : tc_gemm_launch(g, g.a_ms, s);
  return launch_simt_gemm(g, s);
}

}  // namespace

namespace mla {
// Records `msg` as this host thread's mla_last_error() and returns `st`.
mla_status record_error(mla_status st, const char* msg) { return fail(st, "%s", msg); }

mla_status check_dims(const mla_dims* d) {
  REQUIRE(d != nullptr, "dims is NULL");
  REQUIRE(d->n_h > 0 && d->d_h > 0 && d->d_c > 0 && d->d_v > 0 && d->page_size > 0,
          "dims must be positive (n_h=%d d_h=%d d_c=%d d_v=%d page_size=%d)", d->n_h, d->d_h,
          d->d_c, d->d_v, d->page_size);
  REQUIRE(d->d_r >= 0 && d->d_r % 2 == 0, "d_r must be even and >= 0 (got %d)", d->d_r);
  REQUIRE(d->d_model >= 0 && d->d_cq >= 0, "d_model and d_cq must be >= 0");
  return MLA_OK;
}

mla_status check_dtype(int dt) {
  REQUIRE(dt == MLA_F32 || dt == MLA_BF16,
          "dtype %d: this call takes MLA_F32 or MLA_BF16 (the FP8 cache is for decode only)", dt);
  return MLA_OK;
}

mla_status check_decode_dtype(int dt) {
  REQUIRE(dt == MLA_F32 || dt == MLA_BF16 || dt == MLA_FP8_E4M3, "unknown dtype %d", dt);
  return MLA_OK;
}


int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int pick_path(mla_dtype dt, const mla_dims* d) {
  if (g_forced_path == 0) return 0;
  const bool tc_ok = dt == MLA_BF16 && tc_decode_supported(d->n_h, d->d_c, d->d_r, d->page_size);
  if (!tc_ok) return 0;
  return g_forced_path == 2 ? 2 : 1;
}

int plan_unit(int path, int rows, int max_pages, int page_size, int workers) {
  if (path == 0 && page_size > 32 && page_size % 32 == 0 && (long long)rows * max_pages < workers)
    return 32;
  return page_size;
}

int workers_for(int path) {
  const int sms = device_sms();
  if (sms <= 0) return 0;
  if (path == 1) return tc_pair_workers(sms);
  if (path == 2) return tc_split_workers(sms);
  return sms;
}


cudaError_t launch_decode(const DecodeSetup& ds, const void* q_cat, const void* cache,
                          const int32_t* block_table, int max_pages, int num_pages, int B,
                          float softmax_scale, void* ws, float* o_lat, float* lse, mla_dtype dtype,
                          const mla_dims* d, int32_t* dev_status, cudaStream_t s) {
  const int rows = B * ds.q_len;  // query rows
  if (ds.path == 1)
    return tc_pair_launch(q_cat, cache, block_table, max_pages, num_pages, rows, ds.workers,
                          softmax_scale, ws, ds.L, o_lat, lse, dev_status, ds.q_len, s);
  if (ds.path == 2)
    return tc_split_launch(q_cat, cache, block_table, max_pages, num_pages, rows, ds.workers,
                           softmax_scale, ws, ds.L, o_lat, lse, dev_status, ds.q_len, s);
  return launch_simt_decode(q_cat, cache, block_table, max_pages, num_pages, rows, ds.workers,
                            softmax_scale, ws, ds.L, o_lat, lse, d->n_h, d->d_c, d->d_r,
                            d->page_size, ds.unit, dtype == MLA_F32 ? 1 : (dtype == MLA_FP8_E4M3 ? 2 : 0),
                            dev_status, ds.q_len, s);
}

mla_status decode_setup(const void* q_cat, const void* cache, const int32_t* block_table,
                        int max_pages, int num_pages, const int32_t* seq_lens, int B, int q_len,
                        const float* o_lat, const float* lse, mla_dtype dtype,
                        const mla_dims* dims, DecodeSetup* out) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_decode_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0, "B must be >= 0");
  REQUIRE(q_len >= 1 && q_len <= MLA_MAX_NEW_TOKENS, "q_len must be in [1, %d] (got %d)",
          MLA_MAX_NEW_TOKENS, q_len);
  out->path = 0;
  out->workers = 0;
  out->q_len = q_len;
  out->unit = dims->page_size;
  if (B == 0) return MLA_OK;
  REQUIRE(q_cat && cache && block_table && seq_lens && o_lat && lse, "NULL tensor argument");
  REQUIRE(max_pages > 0 && num_pages > 0, "max_pages and num_pages must be > 0");
  REQUIRE(dims->d_c % 32 == 0 && dims->d_c <= 512, "d_c must be a multiple of 32, <= 512");
  out->path = pick_path(dtype, dims);
  out->workers = workers_for(out->path);
  if (out->workers <= 0) return fail(MLA_ERR_CUDA, "cannot query the device's SM count");
  out->unit = plan_unit(out->path, B * q_len, max_pages, dims->page_size, out->workers);
  out->L = workspace_layout(B * q_len, out->workers, dims->n_h, dims->d_c);
  return MLA_OK;
}
}  // namespace mla

extern "C" {

const char* mla_status_string(int st) {
  switch (st) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    default: return "MLA_ERR_UNKNOWN";
  }
}

const char* mla_last_error(void) { return g_last_error.c_str(); }

int mla_abi_version(void) { return MLA_ABI_VERSION; }

void mla_force_decode_path(int path) {
  g_forced_path = (path == 0 || path == 1 || path == 2) ? path : -1;
}

int mla_decode_path(mla_dtype dtype, const mla_dims* dims) {
  if (check_dims(dims) != MLA_OK || check_decode_dtype(dtype) != MLA_OK) return -1;
  return pick_path(dtype, dims);
}

mla_status mla_tc_selftest(const void* q_cat, const void* page, const void* pmat, float* s_out,
                           float* o_out, int half, int32_t* dev_status, void* stream) {
  REQUIRE(q_cat && page && pmat && s_out && o_out, "NULL tensor argument");
  REQUIRE(half == 0 || half == 1, "half must be 0 or 1");
  if (!tc_decode_supported(128, 512, 64, 64))
    return fail(MLA_ERR_UNSUPPORTED, "tensor-core decode kernel needs an sm_103 device");
  return cuda_status(tc_selftest_launch(q_cat, page, pmat, s_out, o_out, half, dev_status, S(stream)),
                     "tc_selftest");
}

mla_status mla_rope_table(float* cos_sin, int max_pos, int d_r, double base, void* stream) {
  REQUIRE(cos_sin != nullptr, "cos_sin is NULL");
  REQUIRE(max_pos >= 0 && d_r > 0 && d_r % 2 == 0, "bad max_pos=%d / d_r=%d", max_pos, d_r);
  REQUIRE(base > 0.0, "base must be > 0");
  return cuda_status(launch_rope_table(cos_sin, max_pos, d_r, base, S(stream)), "rope_table");
}

mla_status mla_append_latent(const void* x, const void* w_dkv_kr, const int32_t* seq_idx,
                             const int32_t* pos, const int32_t* block_table, int B,
                             int max_pages, int num_pages, int T, const float* rope,
                             int max_pos, void* cache, mla_dtype dtype, const mla_dims* dims,
                             int32_t* dev_status, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(T >= 0 && B >= 0, "T and B must be >= 0");
  if (T == 0) return MLA_OK;
  REQUIRE(x && w_dkv_kr && pos && block_table && cache, "NULL tensor argument");
  REQUIRE(dims->d_model > 0, "append needs d_model > 0");
  REQUIRE(B > 0 && max_pages > 0 && num_pages > 0, "B, max_pages, num_pages must be > 0");
  REQUIRE(dims->d_r == 0 || (rope && max_pos > 0), "RoPE table required when d_r > 0");
  const int f32 = dtype == MLA_F32;
  GemmArgs g = {};
  g.a = x; g.a_gs = 0; g.a_ms = dims->d_model; g.a_f32 = f32;
  g.w = w_dkv_kr; g.w_gs = 0; g.w_ns = dims->d_model; g.w_ks = 1; g.w_f32 = f32;
  g.G = 1; g.M = T; g.N = dims->d_c + dims->d_r; g.K = dims->d_model;
  g.epi = EPI_APPEND;
  g.out = cache; g.o_f32 = f32;
  g.rope = rope; g.max_pos = max_pos; g.d_r = dims->d_r; g.rope_off = dims->d_c;
  g.rope_period = g.N; g.pos = pos;
  g.seq_idx = seq_idx; g.block_table = block_table; g.B = B; g.max_pages = max_pages;
  g.num_pages = num_pages; g.page_size = dims->page_size; g.dev_status = dev_status;
  return cuda_status(projection(g, S(stream)), "append_latent");
}

}  // extern "C"

namespace {
// c_Q = x W^DQ^T (or x), then per head [W_up_h] c_Q with RoPE on the last
// d_r of every `per_head` output columns: the query projection (per_head =
// d_h + d_r) or, with the fused W^UK^T W^UQ rows, q_cat itself (per_head =
// d_c + d_r).
mla_status project_query(const void* x, const void* w_dq, const void* w_up, const int32_t* pos,
                         int T, const float* rope, int max_pos, void* c_q, void* out,
                         mla_dtype dtype, const mla_dims* dims, int per_head, int rope_off,
                         int32_t* dev_status, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(T >= 0, "T must be >= 0");
  if (T == 0) return MLA_OK;
  REQUIRE(x && w_up && pos && out, "NULL tensor argument");
  REQUIRE(dims->d_model > 0, "project_q needs d_model > 0");
  REQUIRE(dims->d_cq == 0 || (w_dq && c_q), "d_cq > 0 needs w_dq and the c_q scratch");
  REQUIRE(dims->d_r == 0 || (rope && max_pos > 0), "RoPE table required when d_r > 0");
  const int f32 = dtype == MLA_F32;
  const void* src = x;
  int K = dims->d_model;
  if (dims->d_cq > 0) {
    GemmArgs g = {};
    g.a = x; g.a_ms = dims->d_model; g.a_f32 = f32;
    g.w = w_dq; g.w_ns = dims->d_model; g.w_ks = 1; g.w_f32 = f32;
    g.G = 1; g.M = T; g.N = dims->d_cq; g.K = dims->d_model;
    g.epi = EPI_STORE; g.out = c_q; g.o_ms = dims->d_cq; g.o_f32 = f32;
    if ((st = cuda_status(projection(g, S(stream)), "project_q/W^DQ")) != MLA_OK) return st;
    src = c_q;
    K = dims->d_cq;
  }
  GemmArgs g = {};
  g.a = src; g.a_ms = K; g.a_f32 = f32;
  g.w = w_up; g.w_ns = K; g.w_ks = 1; g.w_f32 = f32;
  g.G = 1; g.M = T; g.N = dims->n_h * per_head; g.K = K;
  g.epi = EPI_ROPE; g.out = out; g.o_ms = g.N; g.o_f32 = f32;
  g.rope = rope; g.max_pos = max_pos; g.d_r = dims->d_r; g.rope_off = rope_off;
  g.rope_period = per_head; g.pos = pos; g.dev_status = dev_status;
  return cuda_status(projection(g, S(stream)), "project_q/up-projection");
}
}  // namespace

extern "C" {

mla_status mla_project_q(const void* x, const void* w_dq, const void* w_uq_qr,
                         const int32_t* pos, int T, const float* rope, int max_pos,
                         void* c_q, void* q, mla_dtype dtype, const mla_dims* dims,
                         int32_t* dev_status, void* stream) {
  if (!dims) return fail(MLA_ERR_INVALID_ARG, "dims is NULL");
  return project_query(x, w_dq, w_uq_qr, pos, T, rope, max_pos, c_q, q, dtype, dims,
                       dims->d_h + dims->d_r, dims->d_h, dev_status, stream);
}

mla_status mla_fuse_query_weights(const void* w_uq_qr, const void* w_uk, void* w_fused_q,
                                  mla_dtype dtype, const mla_dims* dims, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(w_uq_qr && w_uk && w_fused_q, "NULL tensor argument");
  REQUIRE(dims->d_model > 0, "fusing the query weights needs d_model > 0");
  const int f32 = dtype == MLA_F32;
  const int K = dims->d_cq > 0 ? dims->d_cq : dims->d_model;
  const long long in_h = (long long)(dims->d_h + dims->d_r) * K;   // one head of w_uq_qr
  const long long out_h = (long long)(dims->d_c + dims->d_r) * K;  // one head of w_fused_q
  // F_h[c][j] = sum_i W^UK[h d_h + i][c] W^UQ_h[i][j]
  GemmArgs g = {};
  g.a = w_uk; g.a_gs = (long long)dims->d_h * dims->d_c; g.a_ms = 1; g.a_ks = dims->d_c;
  g.a_f32 = f32;
  g.w = w_uq_qr; g.w_gs = in_h; g.w_ns = 1; g.w_ks = K; g.w_f32 = f32;
  g.G = dims->n_h; g.M = dims->d_c; g.N = K; g.K = dims->d_h;
  g.epi = EPI_STORE; g.out = w_fused_q; g.o_gs = out_h; g.o_ms = K; g.o_f32 = f32;
  if ((st = cuda_status(launch_simt_gemm(g, S(stream)), "fuse_query_weights")) != MLA_OK) return st;
  // the W^QR rows of every head follow unchanged
  const int esz = f32 ? 4 : 2;
  const char* src = reinterpret_cast<const char*>(w_uq_qr) + (size_t)dims->d_h * K * esz;
  char* dst = reinterpret_cast<char*>(w_fused_q) + (size_t)dims->d_c * K * esz;
  return cuda_status(launch_copy_rows(src, in_h, K, dst, out_h, K, dims->n_h, dims->d_r, K, esz,
                                      S(stream)),
                     "fuse_query_weights/W^QR");
}

mla_status mla_project_q_absorbed(const void* x, const void* w_dq, const void* w_fused_q,
                                  const int32_t* pos, int T, const float* rope, int max_pos,
                                  void* c_q, void* q_cat, mla_dtype dtype, const mla_dims* dims,
                                  int32_t* dev_status, void* stream) {
  if (!dims) return fail(MLA_ERR_INVALID_ARG, "dims is NULL");
  return project_query(x, w_dq, w_fused_q, pos, T, rope, max_pos, c_q, q_cat, dtype, dims,
                       dims->d_c + dims->d_r, dims->d_c, dev_status, stream);
}

mla_status mla_fuse_output_weights(const void* w_o, const void* w_uv, void* w_fused_o,
                                   mla_dtype dtype, const mla_dims* dims, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(w_o && w_uv && w_fused_o, "NULL tensor argument");
  REQUIRE(dims->d_model > 0, "fusing the output weights needs d_model > 0");
  const int f32 = dtype == MLA_F32;
  // F^O[n][h d_c + c] = sum_v W^O[n][h d_v + v] W^UV[h d_v + v][c]
  GemmArgs g = {};
  g.a = w_o; g.a_gs = dims->d_v; g.a_ms = (long long)dims->n_h * dims->d_v; g.a_ks = 1;
  g.a_f32 = f32;
  g.w = w_uv; g.w_gs = (long long)dims->d_v * dims->d_c; g.w_ns = 1; g.w_ks = dims->d_c;
  g.w_f32 = f32;
  g.G = dims->n_h; g.M = dims->d_model; g.N = dims->d_c; g.K = dims->d_v;
  g.epi = EPI_STORE; g.out = w_fused_o; g.o_gs = dims->d_c;
  g.o_ms = (long long)dims->n_h * dims->d_c; g.o_f32 = f32;
  return cuda_status(launch_simt_gemm(g, S(stream)), "fuse_output_weights");
}

mla_status mla_out_proj_absorbed(const float* o_lat, void* o_lat_lowp, const void* w_fused_o,
                                 float* u, int B, mla_dtype dtype, const mla_dims* dims,
                                 void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0, "B must be >= 0");
  if (B == 0) return MLA_OK;
  REQUIRE(o_lat && w_fused_o && u, "NULL tensor argument");
  REQUIRE(dims->d_model > 0, "out_proj needs d_model > 0");
  const int K = dims->n_h * dims->d_c;
  const void* a = o_lat;
  if (dtype == MLA_BF16) {
    REQUIRE(o_lat_lowp != nullptr, "bf16 weights need the o_lat_lowp scratch");
    if ((st = cuda_status(launch_to_bf16(o_lat, o_lat_lowp, (long long)B * K, S(stream)),
                          "out_proj_absorbed/round")) != MLA_OK)
      return st;
    a = o_lat_lowp;
  }
  GemmArgs g = {};
  g.a = a; g.a_ms = K; g.a_f32 = dtype == MLA_F32;
  g.w = w_fused_o; g.w_ns = K; g.w_ks = 1; g.w_f32 = dtype == MLA_F32;
  g.G = 1; g.M = B; g.N = dims->d_model; g.K = K;
  g.epi = EPI_STORE; g.out = u; g.o_ms = dims->d_model; g.o_f32 = 1;
  return cuda_status(projection(g, S(stream)), "out_proj_absorbed");
}

mla_status mla_gather_latent(const void* cache, const int32_t* block_table, int max_pages,
                             int num_pages, int seq, int n_tokens, void* rows, mla_dtype dtype,
                             const mla_dims* dims, int32_t* dev_status, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(n_tokens >= 0 && seq >= 0, "seq and n_tokens must be >= 0");
  if (n_tokens == 0) return MLA_OK;
  REQUIRE(cache && block_table && rows, "NULL tensor argument");
  REQUIRE(max_pages > 0 && num_pages > 0, "max_pages and num_pages must be > 0");
  REQUIRE(n_tokens <= max_pages * dims->page_size, "n_tokens past the block table");
  const int esz = dtype == MLA_F32 ? 4 : 2;
  REQUIRE(((dims->d_c + dims->d_r) * esz) % 16 == 0, "row width must be a multiple of 16 bytes");
  return cuda_status(launch_gather_rows(cache, block_table, max_pages, num_pages, dims->page_size,
                                        seq, n_tokens, dims->d_c + dims->d_r, esz, rows,
                                        dev_status, S(stream)),
                     "gather_latent");
}

mla_status mla_expand_kv(const void* rows, const void* w_uk, const void* w_uv, void* k_nope,
                         void* v, int n_tokens, mla_dtype dtype, const mla_dims* dims,
                         void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(n_tokens >= 0, "n_tokens must be >= 0");
  if (n_tokens == 0) return MLA_OK;
  REQUIRE(rows && w_uk && w_uv && k_nope && v, "NULL tensor argument");
  const int f32 = dtype == MLA_F32;
  const int W = dims->d_c + dims->d_r;
  // k_nope[t][h*d_h + i] = sum_c rows[t][c] W^UK[h*d_h + i][c], and the same for W^UV
  for (int which = 0; which < 2; ++which) {
    GemmArgs g = {};
    g.a = rows; g.a_ms = W; g.a_f32 = f32;
    g.w = which == 0 ? w_uk : w_uv; g.w_ns = dims->d_c; g.w_ks = 1; g.w_f32 = f32;
    g.G = 1; g.M = n_tokens; g.N = dims->n_h * (which == 0 ? dims->d_h : dims->d_v);
    g.K = dims->d_c;
    g.epi = EPI_STORE; g.out = which == 0 ? k_nope : v; g.o_ms = g.N; g.o_f32 = f32;
    if ((st = cuda_status(projection(g, S(stream)), which == 0 ? "expand_kv/K" : "expand_kv/V")) !=
        MLA_OK)
      return st;
  }
  return MLA_OK;
}

mla_status mla_prefill_attn(const void* q, const void* k_nope, const void* rows, const void* v,
                            void* o, float* lse, int n_tokens, float softmax_scale,
                            mla_dtype dtype, const mla_dims* dims, int32_t* dev_status,
                            void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(n_tokens >= 0, "n_tokens must be >= 0");
  if (n_tokens == 0) return MLA_OK;
  REQUIRE(q && k_nope && rows && v && o, "NULL tensor argument");
  if (dtype != MLA_BF16 ||
      !tc_prefill_supported(dims->n_h, dims->d_h, dims->d_r, dims->d_c, dims->d_v))
    return fail(MLA_ERR_UNSUPPORTED,
                "prefill attention is built for bf16 and n_h=128, d_h=d_v=128, d_r=64, d_c=512 "
                "on an sm_103 device");
  return cuda_status(tc_prefill_launch(q, k_nope, rows, v, o, lse, n_tokens, softmax_scale,
                                       dev_status, S(stream)),
                     "prefill_attn (tcgen05)");
}

mla_status mla_absorb_q(const void* q, const void* w_uk, void* q_cat, int B, mla_dtype dtype,
                        const mla_dims* dims, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0, "B must be >= 0");
  if (B == 0) return MLA_OK;
  REQUIRE(q && w_uk && q_cat, "NULL tensor argument");
  const int f32 = dtype == MLA_F32;
  if (!f32 && g_forced_path != 0 &&
      tc_absorb_supported(dims->n_h, dims->d_h, dims->d_r, dims->d_c, dims->d_v))
    return cuda_status(tc_absorb_q_launch(q, w_uk, q_cat, B, nullptr, S(stream)),
                       "absorb_q (tcgen05)");
  const int qw = dims->d_h + dims->d_r, cw = dims->d_c + dims->d_r;
  GemmArgs g = {};
  g.a = q; g.a_gs = qw; g.a_ms = (long long)dims->n_h * qw; g.a_f32 = f32;
  g.w = w_uk; g.w_gs = (long long)dims->d_h * dims->d_c; g.w_ns = 1; g.w_ks = dims->d_c;
  g.w_f32 = f32;
  g.G = dims->n_h; g.M = B; g.N = dims->d_c; g.K = dims->d_h;
  g.epi = EPI_STORE; g.out = q_cat; g.o_gs = cw; g.o_ms = (long long)dims->n_h * cw; g.o_f32 = f32;
  if ((st = cuda_status(launch_simt_gemm(g, S(stream)), "absorb_q")) != MLA_OK) return st;
  return cuda_status(launch_copy_rope_part(q, q_cat, B, dims->n_h, dims->d_h, dims->d_r,
                                           dims->d_c, f32, S(stream)),
                     "absorb_q/rope part");
}

size_t mla_decode_workspace_size(int B, mla_dtype dtype, const mla_dims* dims) {
  if (check_dims(dims) != MLA_OK || check_decode_dtype(dtype) != MLA_OK || B < 0) return 0;
  const int workers = workers_for(pick_path(dtype, dims));
  if (workers <= 0) return 0;
  return workspace_layout(B, workers, dims->n_h, dims->d_c).total;
}

mla_status mla_plan_decode_mtp(const int32_t* seq_lens, int B, int q_len, int max_pages,
                               void* workspace, size_t ws_bytes, mla_dtype dtype,
                               const mla_dims* dims, int32_t* dev_status, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_decode_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0 && max_pages > 0, "B must be >= 0 and max_pages > 0");
  REQUIRE(q_len >= 1 && q_len <= MLA_MAX_NEW_TOKENS, "q_len must be in [1, %d] (got %d)",
          MLA_MAX_NEW_TOKENS, q_len);
  if (B == 0) return MLA_OK;
  REQUIRE(seq_lens != nullptr, "seq_lens is NULL");
  const int path = pick_path(dtype, dims);
  const int workers = workers_for(path);
  if (workers <= 0) return fail(MLA_ERR_CUDA, "cannot query the device's SM count");
  const WorkspaceLayout L = workspace_layout(B * q_len, workers, dims->n_h, dims->d_c);
  if (!workspace || ws_bytes < L.total)
    return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu required", ws_bytes, L.total);
  const int unit = plan_unit(path, B * q_len, max_pages, dims->page_size, workers);
  return cuda_status(launch_plan(seq_lens, B, q_len, max_pages * (dims->page_size / unit), unit, workers, path,
                                 dtype != MLA_F32, workspace, L, dev_status, S(stream)),
                     "plan_decode");
}

mla_status mla_plan_decode(const int32_t* seq_lens, int B, int max_pages, void* workspace,
                           size_t ws_bytes, mla_dtype dtype, const mla_dims* dims,
                           int32_t* dev_status, void* stream) {
  return mla_plan_decode_mtp(seq_lens, B, 1, max_pages, workspace, ws_bytes, dtype, dims,
                             dev_status, stream);
}

mla_status mla_decode_attn_mtp(const void* q_cat, const void* cache, const int32_t* block_table,
                               int max_pages, int num_pages, const int32_t* seq_lens, int B,
                               int q_len, float softmax_scale, void* workspace, size_t ws_bytes,
                               float* o_lat, float* lse, mla_dtype dtype, const mla_dims* dims,
                               int32_t* dev_status, void* stream) {
  DecodeSetup ds;
  mla_status st = decode_setup(q_cat, cache, block_table, max_pages, num_pages, seq_lens, B, q_len,
                               o_lat, lse, dtype, dims, &ds);
  if (st != MLA_OK || B == 0) return st;
  if (!workspace || ws_bytes < ds.L.total)
    return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu required", ws_bytes, ds.L.total);
  // the plan in the workspace carries the validated lengths
  return cuda_status(launch_decode(ds, q_cat, cache, block_table, max_pages, num_pages, B,
                                   softmax_scale, workspace, o_lat, lse, dtype, dims, dev_status,
                                   S(stream)),
                     ds.path == 0 ? "decode_attn (simt)" : "decode_attn (tcgen05)");
}

mla_status mla_decode_attn(const void* q_cat, const void* cache, const int32_t* block_table,
                           int max_pages, int num_pages, const int32_t* seq_lens, int B,
                           float softmax_scale, void* workspace, size_t ws_bytes, float* o_lat,
                           float* lse, mla_dtype dtype, const mla_dims* dims,
                           int32_t* dev_status, void* stream) {
  return mla_decode_attn_mtp(q_cat, cache, block_table, max_pages, num_pages, seq_lens, B, 1,
                             softmax_scale, workspace, ws_bytes, o_lat, lse, dtype, dims,
                             dev_status, stream);
}

mla_status mla_combine(const void* workspace, size_t ws_bytes, int B, float* o_lat, float* lse,
                       mla_dtype dtype, const mla_dims* dims, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_decode_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0, "B must be >= 0");
  if (B == 0) return MLA_OK;
  REQUIRE(o_lat && lse, "NULL tensor argument");
  const int workers = workers_for(pick_path(dtype, dims));
  if (workers <= 0) return fail(MLA_ERR_CUDA, "cannot query the device's SM count");
  const WorkspaceLayout L = workspace_layout(B, workers, dims->n_h, dims->d_c);
  if (!workspace || ws_bytes < L.total)
    return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu required", ws_bytes, L.total);
  return cuda_status(launch_combine(workspace, L, B, dims->n_h, dims->d_c, o_lat, lse, S(stream)),
                     "combine");
}

mla_status mla_absorb_out(const float* o_lat, const void* w_uv, void* o, int B, mla_dtype dtype,
                          mla_dtype out_dtype, const mla_dims* dims, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  if ((st = check_dtype(out_dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0, "B must be >= 0");
  if (B == 0) return MLA_OK;
  REQUIRE(o_lat && w_uv && o, "NULL tensor argument");
  if (dtype == MLA_BF16 && g_forced_path != 0 &&
      tc_absorb_supported(dims->n_h, dims->d_h, dims->d_r, dims->d_c, dims->d_v))
    return cuda_status(tc_absorb_out_launch(o_lat, w_uv, o, out_dtype == MLA_F32, B, nullptr,
                                            S(stream)),
                       "absorb_out (tcgen05)");
  GemmArgs g = {};
  g.a = o_lat; g.a_gs = dims->d_c; g.a_ms = (long long)dims->n_h * dims->d_c; g.a_f32 = 1;
  g.w = w_uv; g.w_gs = (long long)dims->d_v * dims->d_c; g.w_ns = dims->d_c; g.w_ks = 1;
  g.w_f32 = dtype == MLA_F32;
  g.G = dims->n_h; g.M = B; g.N = dims->d_v; g.K = dims->d_c;
  g.epi = EPI_STORE; g.out = o; g.o_gs = dims->d_v; g.o_ms = (long long)dims->n_h * dims->d_v;
  g.o_f32 = out_dtype == MLA_F32;
  return cuda_status(launch_simt_gemm(g, S(stream)), "absorb_out");
}

mla_status mla_combine_absorb_out(const void* workspace, size_t ws_bytes, int B, float* o_lat,
                                  float* lse, const void* w_uv, void* o, mla_dtype dtype,
                                  mla_dtype out_dtype, const mla_dims* dims, int32_t* dev_status,
                                  void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  if ((st = check_dtype(out_dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0, "B must be >= 0");
  if (B == 0) return MLA_OK;
  REQUIRE(o_lat && lse && w_uv && o, "NULL tensor argument");
  const int path = pick_path(dtype, dims);
  const int workers = workers_for(path);
  if (workers <= 0) return fail(MLA_ERR_CUDA, "cannot query the device's SM count");
  const WorkspaceLayout L = workspace_layout(B, workers, dims->n_h, dims->d_c);
  if (!workspace || ws_bytes < L.total)
    return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu required", ws_bytes, L.total);
  if (dtype == MLA_BF16 && g_forced_path != 0 &&
      tc_absorb_supported(dims->n_h, dims->d_h, dims->d_r, dims->d_c, dims->d_v))
    return cuda_status(tc_absorb_out_merge_launch(workspace, L, o_lat, lse, w_uv, o,
                                                  out_dtype == MLA_F32, B, dev_status, S(stream)),
                       "combine_absorb_out (tcgen05)");
  if ((st = mla_combine(workspace, ws_bytes, B, o_lat, lse, dtype, dims, stream)) != MLA_OK) return st;
  return mla_absorb_out(o_lat, w_uv, o, B, dtype, out_dtype, dims, stream);
}

mla_status mla_out_proj(const void* o, const void* w_o, float* u, int B, mla_dtype dtype,
                        const mla_dims* dims, void* stream) {
  mla_status st = check_dims(dims);
  if (st != MLA_OK) return st;
  if ((st = check_dtype(dtype)) != MLA_OK) return st;
  REQUIRE(B >= 0, "B must be >= 0");
  if (B == 0) return MLA_OK;
  REQUIRE(o && w_o && u, "NULL tensor argument");
  REQUIRE(dims->d_model > 0, "out_proj needs d_model > 0");
  const int K = dims->n_h * dims->d_v;
  GemmArgs g = {};
  g.a = o; g.a_ms = K; g.a_f32 = dtype == MLA_F32;
  g.w = w_o; g.w_ns = K; g.w_ks = 1; g.w_f32 = dtype == MLA_F32;
  g.G = 1; g.M = B; g.N = dims->d_model; g.K = K;
  g.epi = EPI_STORE; g.out = u; g.o_ms = dims->d_model; g.o_f32 = 1;
  return cuda_status(projection(g, S(stream)), "out_proj");
}

}  // extern "C"
