// Device router: f32 logits GEMV + sigmoid + bias (every CTA), then bias-augmented top-K
// selection, raw-score weights, top-p, norm_topk and routed_scale (the CTA that finishes last).
//
// c/backend_cuda.cu commit history, commit "First increment of the #431 plan": an E x D f32
// logits GEMV + sigmoid, then a selection step that does bias-augmented top-K by choice with a
// strict '>' tie-break, weights from the raw score, route-level TOPP truncation, norm_topk and
// routed_scale. For S > 1 the logits of all tokens come from one launch (the batched router of
// the "GPU resident pipeline" commit).
#include <mutex>
#include <string>

#include "coli_internal.h"
#include "pipe.h"

namespace coli {

#ifndef COLI_ROUTER_THREADS
#define COLI_ROUTER_THREADS 256
#endif
#ifndef COLI_ROUTER_UNROLL
#define COLI_ROUTER_UNROLL 4
#endif
constexpr int kRouterThreads = COLI_ROUTER_THREADS;
constexpr int kRouterUnroll = COLI_ROUTER_UNROLL;  // float4 loads of one thread in flight together
#ifndef COLI_ROUTER_ROWS
#define COLI_ROUTER_ROWS 1
#endif
constexpr int kRowsPerCta = COLI_ROUTER_ROWS;  // E = 256 -> 256 CTAs, every row in flight at once

// Order-preserving map of a finite binary32 value to uint32 (larger float -> larger integer;
// -0 is folded onto +0 so that the two compare equal, as floats do).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void select_finish(int mine, float wmine, int K, float topp, int norm_topk,
                                              float routed_scale, int shared, int32_t* __restrict__ idx_out,
                                              float* __restrict__ w_out, int32_t* __restrict__ nsel_out,
                                              const ExpertDesc* table);

// One warp selects for one token. Lane l owns experts e = l + 32 * i (i < EPL). Each round, every
// lane finds its best not-yet-chosen expert by a strict '>' scan in increasing e (so its first,
// lowest index wins a local tie); the warp maximum of the order keys and then the minimum index
// among the lanes holding that maximum are taken with warp reductions, so a tie across lanes also
// goes to the lower index. The chosen expert's raw score travels with it.
template <int EPL>
__device__ void select_token(const float2* __restrict__ sc_row, int E, int K, float topp, int norm_topk,
                             float routed_scale, int shared, int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                             int32_t* __restrict__ nsel_out, int* err, const ExpertDesc* table) {
  const int lane = threadIdx.x & 31;
  uint32_t key[EPL];
  float sv[EPL];
  unsigned taken = 0;  // bit i: expert lane + 32 i already chosen (or absent)
  bool bad = false;
#pragma unroll
  for (int i = 0; i < EPL; i++) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float2 v = __ldcg(sc_row + e);  // (score, choice)
      if (!isfinite(v.x) || !isfinite(v.y)) bad = true;
      key[i] = order_key(v.y);
      sv[i] = v.x;
    } else {
      key[i] = 0;
      sv[i] = 0.f;
      taken |= 1u << i;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, COLI_E_NONFINITE);
  int mine = -1;      // lane k keeps the expert chosen in round k ...
  float wmine = 0.f;  // ... and its raw score
  for (int k = 0; k < K; k++) {
    uint32_t bk = 0;
    int bi = -1;
    float bs = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
      if (!(taken & (1u << i)) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = i;
        bs = sv[i];
      }
    }
    const uint32_t best = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t cand = (bi >= 0 && bk == best) ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    const float ws = __shfl_sync(0xffffffffu, bs, win & 31);
    if ((int)(win & 31) == lane) taken |= 1u << (win >> 5);
    if (lane == k) {
      mine = (int)win;
      wmine = ws;
    }
  }
  select_finish(mine, wmine, K, topp, norm_topk, routed_scale, shared, idx_out, w_out, nsel_out, table);
}

// Lane k holds the expert of slot k (mine) and its raw score (wmine): weights from the raw
// (bias-free) score, top-p, norm and scale; every sum in slot order in binary32, no contraction.
__device__ __forceinline__ void select_finish(int mine, float wmine, int K, float topp, int norm_topk,
                                              float routed_scale, int shared, int32_t* __restrict__ idx_out,
                                              float* __restrict__ w_out, int32_t* __restrict__ nsel_out,
                                              const ExpertDesc* table) {
  const int lane = threadIdx.x & 31;
  int m = K;
  float denom = 1.f;
  float total = 0.f;
  for (int k = 0; k < K; k++) total = __fadd_rn(total, __shfl_sync(0xffffffffu, wmine, k));
  if (topp > 0.f && topp < 1.f) {
    float cum = 0.f;
    for (int k = 0; k < K; k++) {
      cum = __fadd_rn(cum, __fdiv_rn(__shfl_sync(0xffffffffu, wmine, k), total));
      if (cum >= topp) {
        m = k + 1;
        break;
      }
    }
  }
  if (norm_topk) {
    denom = 0.f;
    for (int k = 0; k < m; k++) denom = __fadd_rn(denom, __shfl_sync(0xffffffffu, wmine, k));
  }
  // shared >= 0: the shared expert follows the kept slots as one more kept slot of weight 1 (no
  // normalisation, no routed scale), and the row has K + 1 slots
  const bool has_shared = shared >= 0;
  if (lane < K + has_shared) {
    const bool kept = lane < m;
    const bool is_shared = has_shared && lane == m;
    const float wv = norm_topk ? __fdiv_rn(wmine, denom) : wmine;
    idx_out[lane] = kept ? mine : (is_shared ? shared : -1);
    w_out[lane] = kept ? __fmul_rn(wv, routed_scale) : (is_shared ? 1.0f : 0.f);
  }
  if (lane == 0 && nsel_out) *nsel_out = m + has_shared;
  // The chosen experts' table entries go to L2: the expert kernels that follow read them first
  // (a hint only; every id below E, and the shared id, is inside the table).
  const int pe = lane < K ? mine : (has_shared && lane == K ? shared : -1);
  if (table && pe >= 0)
    for (int l = 0; l < (int)(sizeof(ExpertDesc) / 128); l++)
      prefetch_l2_line(reinterpret_cast<const char*>(table + pe) + 128 * l);
}

// Selection for 1024 < E <= COLI_MAX_EXPERTS (more than 32 experts per lane): the same rules and
// reductions as select_token, but each round re-reads the lane's (score, choice) pairs through L2
// instead of holding them in registers, and the chosen set is a 128-bit mask per lane.
__device__ void select_token_large(const float2* __restrict__ sc_row, int E, int K, float topp, int norm_topk,
                                   float routed_scale, int shared, int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                   int32_t* __restrict__ nsel_out, int* err, const ExpertDesc* table) {
  const int lane = threadIdx.x & 31;
  const int epl = (E + 31) >> 5;           // <= 128
  uint32_t taken[4] = {0u, 0u, 0u, 0u};   // bit i: expert lane + 32 i already chosen (or absent)
  bool bad = false;
  for (int i = 0; i < epl; i++) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float2 v = __ldcg(sc_row + e);
      if (!isfinite(v.x) || !isfinite(v.y)) bad = true;
    } else {
      taken[i >> 5] |= 1u << (i & 31);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, COLI_E_NONFINITE);
  int mine = -1;
  float wmine = 0.f;
  for (int k = 0; k < K; k++) {
    uint32_t bk = 0;
    int bi = -1;
    float bs = 0.f;
    for (int i = 0; i < epl; i++) {
      if (taken[i >> 5] & (1u << (i & 31))) continue;
      const float2 v = __ldcg(sc_row + lane + 32 * i);
      const uint32_t key = order_key(v.y);
      if (bi < 0 || key > bk) {
        bk = key;
        bi = i;
        bs = v.x;
      }
    }
    const uint32_t best = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t cand = (bi >= 0 && bk == best) ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    const float ws = __shfl_sync(0xffffffffu, bs, win & 31);
    if ((int)(win & 31) == lane) taken[(win >> 5) >> 5] |= 1u << ((win >> 5) & 31);
    if (lane == k) {
      mine = (int)win;
      wmine = ws;
    }
  }
  select_finish(mine, wmine, K, topp, norm_topk, routed_scale, shared, idx_out, w_out, nsel_out, table);
}

// EPL = experts per lane (a power of two up to 32); EPL = 0: the large-E selection.
template <int EPL>
__device__ __forceinline__ void select_token_any(const float2* sc_row, int E, int K, float topp, int norm_topk,
                                                 float routed_scale, int shared, int32_t* idx_out, float* w_out,
                                                 int32_t* nsel_out, int* err, const ExpertDesc* table) {
  if constexpr (EPL == 0)
    select_token_large(sc_row, E, K, topp, norm_topk, routed_scale, shared, idx_out, w_out, nsel_out, err, table);
  else
    select_token<EPL>(sc_row, E, K, topp, norm_topk, routed_scale, shared, idx_out, w_out, nsel_out, err, table);
}

template <int EPL>
__device__ void select_all(const float2* sc, int S, int E, int K, float topp, int norm_topk, float routed_scale,
                           int shared, int32_t* idx, float* w, int32_t* n_sel, int* err, const ExpertDesc* table) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int slots = K + (shared >= 0);  // output slots per token
  for (int t = warp; t < S; t += nwarps)
    select_token_any<EPL>(sc + (size_t)t * E, E, K, topp, norm_topk, routed_scale, shared, idx + (size_t)t * slots,
                          w + (size_t)t * slots, n_sel ? n_sel + t : nullptr, err, table);
}

// Logits GEMV: CTA b computes rows e = b * kRowsPerCta + r (r < kRowsPerCta) for every token;
// thread t accumulates columns t, t + kRouterThreads, ... (float4 when aligned) for all rows at
// once, so all of a row group's loads are in flight together.
// `status` is the context's error word; `arrivals` counts the CTAs that have stored their scores
// (zero on entry, reset to zero by the CTA that finishes last).
template <bool VEC4>
__device__ __forceinline__ void router_body(const void* __restrict__ x, int x_dtype, int S, int D,
                                            const float* __restrict__ Wr, const float* __restrict__ bias, int E,
                                            int K, float topp, int norm_topk, float routed_scale, int shared,
                                            float2* __restrict__ sc_ws, int32_t* __restrict__ idx,
                                            float* __restrict__ w, int32_t* __restrict__ n_sel,
                                            int* __restrict__ status, unsigned* arrivals, int epl,
                                            const ExpertDesc* table) {
  __shared__ float red[kRouterThreads / 32][kRowsPerCta];
  __shared__ int am_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e0 = blockIdx.x * kRowsPerCta;
  const int nrows = min(kRowsPerCta, E - e0);
  griddep_wait();               // x may be the previous kernel's output
  griddep_launch_dependents();  // the gate/up kernel may start its prologue
  for (int t = 0; t < S; t++) {
    float acc[kRowsPerCta];
#pragma unroll
    for (int r = 0; r < kRowsPerCta; r++) acc[r] = 0.f;
    if (VEC4 && x_dtype == COLI_DTYPE_F32) {
      const float4* x4 = reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)t * D);
#pragma unroll kRouterUnroll
      for (int j = tid; j < D / 4; j += kRouterThreads) {
        const float4 b = __ldg(x4 + j);
#pragma unroll
        for (int r = 0; r < kRowsPerCta; r++) {
          if (r < nrows) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(Wr + (size_t)(e0 + r) * D) + j);
            acc[r] = fmaf(a.x, b.x, acc[r]);
            acc[r] = fmaf(a.y, b.y, acc[r]);
            acc[r] = fmaf(a.z, b.z, acc[r]);
            acc[r] = fmaf(a.w, b.w, acc[r]);
          }
        }
      }
    } else {
#pragma unroll 4
      for (int j = tid; j < D; j += kRouterThreads) {
        const float b = load_act(x, x_dtype, (size_t)t * D + j);
#pragma unroll
        for (int r = 0; r < kRowsPerCta; r++)
          if (r < nrows) acc[r] = fmaf(__ldg(Wr + (size_t)(e0 + r) * D + j), b, acc[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerCta; r++) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
      if (lane == 0) red[warp][r] = acc[r];
    }
    __syncthreads();
    if (tid < nrows) {
      float z = 0.f;
      for (int i = 0; i < kRouterThreads / 32; i++) z += red[i][tid];
      const int e = e0 + tid;
      const float sc = 1.0f / (1.0f + expf(-z));
      const float ch = bias ? __fadd_rn(sc, __ldg(bias + e)) : sc;
      sc_ws[(size_t)t * E + e] = make_float2(sc, ch);
    }
    __syncthreads();
  }
  // The CTA that finishes last runs the selection over every token's complete score row.
  // (the arrival is a release of this CTA's stores, ordered after them by the barrier above, and
  // for the last CTA an acquire of every other CTA's)
  if (tid == 0) {
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(prev) : "l"(arrivals) : "memory");
    am_last = prev == gridDim.x - 1;
  }
  __syncthreads();
  if (!am_last) return;
  switch (epl) {
    case 1: select_all<1>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel, status, table); break;
    case 2: select_all<2>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel, status, table); break;
    case 4: select_all<4>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel, status, table); break;
    case 8: select_all<8>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel, status, table); break;
    case 16: select_all<16>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel, status, table); break;
    default: select_all<32>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel, status, table); break;
  }
  __syncthreads();
  if (tid == 0) atomicExch(arrivals, 0u);
}

template <bool VEC4>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(
    const void* __restrict__ x, int x_dtype, int S, int D, const float* __restrict__ Wr,
    const float* __restrict__ bias, int E, int K, float topp, int norm_topk, float routed_scale, int shared,
    float2* __restrict__ sc_ws, int32_t* __restrict__ idx, float* __restrict__ w,
    int32_t* __restrict__ n_sel, int* __restrict__ status, int epl, const ExpertDesc* table) {
  router_body<VEC4>(x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, sc_ws, idx, w, n_sel, status,
                    reinterpret_cast<unsigned*>(status + 1), epl, table);
}

template <bool VEC4>
__global__ void __launch_bounds__(kRouterThreads) router_fixed_kernel(
    const void* __restrict__ x, int x_dtype, int S, int D, const float* __restrict__ Wr,
    const float* __restrict__ bias, int E, int K, float topp, int norm_topk, float routed_scale, int shared,
    float2* __restrict__ sc_ws, int32_t* __restrict__ idx, float* __restrict__ w,
    int32_t* __restrict__ n_sel, int* __restrict__ status, unsigned* arrivals, int epl, const ExpertDesc* table) {
  router_body<VEC4>(x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, sc_ws, idx, w, n_sel, status,
                    arrivals, epl, table);
}

// ------------------------------------------------------------------------------------------
// Many tokens (S >= kBatchedS): the logits as a tiled f32 GEMM, each CTA a 64-token x 64-expert
// tile over one of kRSplit column ranges of D; the ranges are summed in a fixed order, then
// sigmoid and bias give the (score, choice) pairs and one warp per token selects.
// ------------------------------------------------------------------------------------------

constexpr int kBatchedS = 16;
// The decode router's last-CTA selection holds at most 32 experts per lane (E <= 1024); larger E
// takes the many-token path, whose separate selection kernel also has the large-E form.
constexpr int kDecodeMaxE = 1024;
constexpr int kRT = 64;     // tokens and experts per tile
constexpr int kRBK = 32;    // columns of D per step
constexpr int kRSplit = 8;  // column ranges of D

__global__ void __launch_bounds__(256) router_gemm_kernel(const void* __restrict__ x, int x_dtype, int S, int D,
                                                          const float* __restrict__ Wr, int E, float* __restrict__ part) {
  __shared__ __align__(16) float xs[kRBK][kRT + 4];  // [column][token]
  __shared__ __align__(16) float ws[kRBK][kRT + 4];  // [column][expert]
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;  // thread: tokens 4 ty .., experts 4 tx ..
  const int e0 = blockIdx.x * kRT, s0 = blockIdx.y * kRT;
  const int per = ((D + kRSplit - 1) / kRSplit + kRBK - 1) / kRBK * kRBK;
  const int d0 = blockIdx.z * per, d1 = min(D, d0 + per);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
  // thread loads 8 elements of each tile per step: row (i / kRBK), column (i % kRBK), i = tid + 256 m
  float px[8], pw[8];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int m = 0; m < 8; m++) {
      const int i = tid + 256 * m, r = i / kRBK, k = k0 + i % kRBK;
      px[m] = (s0 + r < S && k < d1) ? load_act(x, x_dtype, (size_t)(s0 + r) * D + k) : 0.f;
      pw[m] = (e0 + r < E && k < d1) ? __ldg(Wr + (size_t)(e0 + r) * D + k) : 0.f;
    }
  };
  if (d0 < d1) fetch(d0);
  for (int k0 = d0; k0 < d1; k0 += kRBK) {
#pragma unroll
    for (int m = 0; m < 8; m++) {
      const int i = tid + 256 * m;
      xs[i % kRBK][i / kRBK] = px[m];
      ws[i % kRBK][i / kRBK] = pw[m];
    }
    __syncthreads();
    if (k0 + kRBK < d1) fetch(k0 + kRBK);  // the next step's loads overlap this step's FMAs
#pragma unroll 8
    for (int kk = 0; kk < kRBK; kk++) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[kk][4 * ty]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[kk][4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int s = s0 + 4 * ty + i, e = e0 + 4 * tx + j;
      if (s < S && e < E) part[((size_t)blockIdx.z * S + s) * E + e] = acc[i][j];
    }
}

__global__ void router_finish_kernel(const float* __restrict__ part, int S, int E, const float* __restrict__ bias,
                                     float2* __restrict__ sc_ws) {
  const long long n = (long long)S * E;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    float z = 0.f;
    for (int sp = 0; sp < kRSplit; sp++) z += part[(size_t)sp * n + i];
    const int e = (int)(i % E);
    const float sc = 1.0f / (1.0f + expf(-z));
    sc_ws[i] = make_float2(sc, bias ? __fadd_rn(sc, __ldg(bias + e)) : sc);
  }
}

template <int EPL>
__global__ void router_select_kernel(const float2* sc, int S, int E, int K, float topp, int norm_topk,
                                     float routed_scale, int shared, int32_t* idx, float* w, int32_t* n_sel, int* err,
                                     const ExpertDesc* table) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= S) return;  // uniform per warp
  const int slots = K + (shared >= 0);  // output slots per token
  select_token_any<EPL>(sc + (size_t)t * E, E, K, topp, norm_topk, routed_scale, shared, idx + (size_t)t * slots,
                        w + (size_t)t * slots, n_sel ? n_sel + t : nullptr, err, table);
}

// sc_ws: S E (score, choice) pairs; part: kRSplit S E floats
static int launch_router_batched(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                                 const float* bias, int E, int K, float topp, int norm_topk, float routed_scale,
                                 int shared, int32_t* idx, float* w, int32_t* n_sel, float2* sc_ws, float* part) {
  const ExpertDesc* table = ctx->table_count > 0 ? ctx->d_table : nullptr;
  ProfScope prof(ctx, COLI_KERNEL_ROUTER);
  router_gemm_kernel<<<dim3((E + kRT - 1) / kRT, (S + kRT - 1) / kRT, kRSplit), 256, 0, ctx->stream>>>(x, x_dtype, S, D,
                                                                                                     Wr, E, part);
  const long long n = (long long)S * E;
  int g = (int)((n + 255) / 256);
  if (g > 4 * ctx->num_sms) g = 4 * ctx->num_sms;
  router_finish_kernel<<<g, 256, 0, ctx->stream>>>(part, S, E, bias, sc_ws);
  int epl = 1;
  while (32 * epl < E) epl *= 2;
  const int sg = (S + 7) / 8;
  switch (epl) {
#define COLI_SELECT_CASE(N)                                                                                        \
  case N:                                                                                                          \
    router_select_kernel<N><<<sg, 256, 0, ctx->stream>>>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared,   \
                                                         idx, w, n_sel, ctx->d_status, table);                    \
    break;
    COLI_SELECT_CASE(1)
    COLI_SELECT_CASE(2)
    COLI_SELECT_CASE(4)
    COLI_SELECT_CASE(8)
    COLI_SELECT_CASE(16)
    COLI_SELECT_CASE(32)
    default:  // more than 1024 experts
      router_select_kernel<0><<<sg, 256, 0, ctx->stream>>>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, idx, w,
                                                            n_sel, ctx->d_status, table);
#undef COLI_SELECT_CASE
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "batched router launch");
  return COLI_OK;
}

int launch_router(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr, const float* bias,
                  int E, int K, float topp, int norm_topk, float routed_scale, int shared, int32_t* idx, float* w,
                  int32_t* n_sel) {
  if (S >= kBatchedS || E > kDecodeMaxE) {
    const size_t sc_bytes = align_up((size_t)S * E * sizeof(float2), 256);
    int rc = ensure_workspace(ctx, sc_bytes + (size_t)kRSplit * S * E * sizeof(float));
    if (rc != COLI_OK) return rc;
    return launch_router_batched(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel,
                                 reinterpret_cast<float2*>(ctx->ws.base),
                                 reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ctx->ws.base) + sc_bytes));
  }
  int rc = ensure_workspace(ctx, align_up((size_t)S * E * sizeof(float2), 256));
  if (rc != COLI_OK) return rc;
  float2* sc_ws = reinterpret_cast<float2*>(ctx->ws.base);
  int epl = 1;
  while (32 * epl < E) epl *= 2;
  bool vec4 = (D % 4 == 0) && ((reinterpret_cast<uintptr_t>(Wr) & 15) == 0) &&
              ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
  int grid = (E + kRowsPerCta - 1) / kRowsPerCta;
  ProfScope prof(ctx, COLI_KERNEL_ROUTER);
  const ExpertDesc* table = ctx->table_count > 0 ? ctx->d_table : nullptr;  // for the L2 prefetch hint
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouterThreads);
  cfg.stream = ctx->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* xp = x;
  cudaError_t le = vec4 ? cudaLaunchKernelEx(&cfg, router_kernel<true>, xp, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk,
                                             routed_scale, shared, sc_ws, idx, w, n_sel, ctx->d_status, epl, table)
                        : cudaLaunchKernelEx(&cfg, router_kernel<false>, xp, x_dtype, S, D, Wr, bias, E, K, topp,
                                             norm_topk, routed_scale, shared, sc_ws, idx, w, n_sel, ctx->d_status, epl, table);
  if (le != cudaSuccess) return cuda_fail(ctx, le, "router launch");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "router launch");
  return COLI_OK;
}

// ------------------------------------------------------------------------------------------
// Router entry that allocates nothing (coli_router_select_noalloc).
//
// Some callers cannot let a call allocate device memory: a server that has handed all free HBM to
// its own caching pool (a cudaMalloc would fail or force it to evict), or a decode loop that must
// not stall, since cudaMalloc may synchronise the device and a workspace that grows waits for the
// context's stream first. This entry therefore keeps its scratch in a fixed file-scope device
// array instead of the context's workspace: the arrival counter in the first 256 bytes, then the
// (score, choice) pairs of at most kFixedRouterCells (token, expert) cells, then the partial
// logits of the many-token path. Its address is looked
// up once per device and CUDA context (the first call there), since a device reset or another
// context loads the module at a new address; the counter is cleared on the stream before every
// launch. All contexts on a device share the array, so calls whose kernels could overlap
// (different streams, contexts or host threads without ordering) race on it.
// ------------------------------------------------------------------------------------------

constexpr int kFixedRouterCells = 65536;  // S * E limit
constexpr int kFixedMaxDevices = 64;
// counter (256 B), pairs (512 KiB), partial logits of the many-token path (2 MiB)
constexpr size_t kFixedPairsOff = 256;
constexpr size_t kFixedPartOff = kFixedPairsOff + (size_t)kFixedRouterCells * sizeof(float2);
static __device__ __align__(256) unsigned char
    g_router_fixed[kFixedPartOff + (size_t)kRSplit * kFixedRouterCells * sizeof(float)];

static std::mutex g_fixed_mu;
static unsigned char* g_fixed_addr[kFixedMaxDevices];  // device address of g_router_fixed, once set up ...
static void* g_fixed_ctx[kFixedMaxDevices];            // ... in this CUDA context

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The calling thread's current CUDA context (the primary context of the current device for runtime
// users), through the runtime's driver entry point; NULL if unavailable.
static void* current_context() {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    (void)cudaGetLastError();
  }
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

int launch_router_noalloc(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                          const float* bias, int E, int K, float topp, int norm_topk, float routed_scale,
                          int shared, int32_t* idx, float* w, int32_t* n_sel) {
  if ((long long)S * E > kFixedRouterCells)
    return fail(ctx, COLI_E_INVAL,
                "router_select_noalloc: S * E = " + std::to_string((long long)S * E) + " exceeds the fixed scratch limit " +
                    std::to_string(kFixedRouterCells));
  if (ctx->device < 0 || ctx->device >= kFixedMaxDevices)
    return fail(ctx, COLI_E_INVAL, "router_select_noalloc: device ordinal beyond the fixed scratch table");
  unsigned char* base;
  {
    std::lock_guard<std::mutex> lock(g_fixed_mu);
    void* cur = current_context();  // the caller has made ctx->device current
    base = g_fixed_addr[ctx->device];
    if (!base || g_fixed_ctx[ctx->device] != cur) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_router_fixed);
      if (e != cudaSuccess || !p) return cuda_fail(ctx, e != cudaSuccess ? e : cudaErrorInvalidSymbol, "router_select_noalloc: scratch address");
      base = static_cast<unsigned char*>(p);
      g_fixed_addr[ctx->device] = base;
      g_fixed_ctx[ctx->device] = cur;
    }
  }
  unsigned* arrivals = reinterpret_cast<unsigned*>(base);
  float2* sc_ws = reinterpret_cast<float2*>(base + kFixedPairsOff);
  if (S >= kBatchedS || E > kDecodeMaxE)  // the many-token path, as coli_router_select takes it (no arrival counter)
    return launch_router_batched(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel,
                                 sc_ws, reinterpret_cast<float*>(base + kFixedPartOff));
  cudaError_t e = cudaMemsetAsync(arrivals, 0, sizeof(unsigned), ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "router_select_noalloc: clear counter");
  int epl = 1;
  while (32 * epl < E) epl *= 2;
  const bool vec4 = (D % 4 == 0) && ((reinterpret_cast<uintptr_t>(Wr) & 15) == 0) &&
                    ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
  const int grid = (E + kRowsPerCta - 1) / kRowsPerCta;
  const ExpertDesc* table = ctx->table_count > 0 ? ctx->d_table : nullptr;  // for the L2 prefetch hint
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouterThreads);
  cfg.stream = ctx->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* xp = x;
  ProfScope prof(ctx, COLI_KERNEL_ROUTER);
  e = vec4 ? cudaLaunchKernelEx(&cfg, router_fixed_kernel<true>, xp, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk,
                                routed_scale, shared, sc_ws, idx, w, n_sel, ctx->d_status, arrivals, epl, table)
           : cudaLaunchKernelEx(&cfg, router_fixed_kernel<false>, xp, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk,
                                routed_scale, shared, sc_ws, idx, w, n_sel, ctx->d_status, arrivals, epl, table);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "router_select_noalloc launch");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "router_select_noalloc launch");
  return COLI_OK;
}

}  // namespace coli
