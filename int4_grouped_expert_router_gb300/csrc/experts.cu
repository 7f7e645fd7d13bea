// Grouped int4 expert FFN for decode: fused gate+up dual GEMV with the SiLU(gate)*up epilogue,
// then the down GEMV with per-expert weighting and a fixed-order, atomics-free reduce into the
// residual.
//
// Sources: c/backend_cuda.cu commit history -- commit "The TC_W4A16 branch ..." (the grouped
// 3-launch decode path: dual gate/up GEMV, SiLU, down GEMV), commit "grouped MoE kernels were
// per-row-only" (per-group scales applied inside the accumulation, gs even, gs = 0 per-row,
// mixed members in one launch); PR #434 "COLI_CUDA_RESID=1", section "What" (per-expert
// weighting and fixed-order reduce on the device).
//
// Dot-product arithmetic. A thread owns one 16-byte chunk of a weight row (32 columns) and keeps
// the matching 32 activations in registers in block-fixed-point form: the chunk is scaled by a
// power of two 2^q so that its largest magnitude lies in [2^29, 2^30), rounded to integers and
// split into four balanced signed bytes (x = l3 2^24 + l2 2^16 + l1 2^8 + l0). The nibble-by-limb
// products are then summed exactly in 32-bit integers with dp4a (four products per
// instruction), the offset 8 is removed through a precomputed -8 * sum(l), and the four exact
// limb sums are combined in binary32 and scaled back by 2^-q. The chunk result therefore differs
// from the exact dot product of the given activations by at most one rounding of the final sum
// plus the activation quantisation (below 2^-30 of the chunk's largest activation, per column).
// Chunk results are summed across the warp by a butterfly and across warps in a fixed order.
#include "coli_internal.h"

namespace coli {

// ------------------------------------------------------------------------------------------
// Block-fixed-point activations and the chunk dot product
// ------------------------------------------------------------------------------------------

struct Limbs {
  uint32_t r[4][2][4];  // [16-bit word of the chunk][even/odd columns][limb]: 4 bytes each
  int32_t off[4];       // -8 * sum over the chunk of limb l
  float kf[4];          // 2^(8 l - q)
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// v[j] = activation of column 32 c + j (0 beyond the matrix). Returns false if any is not finite.
__device__ __forceinline__ bool make_limbs(const float (&v)[32], Limbs& L) {
  float M = 0.f;
  bool finite = true;
#pragma unroll
  for (int j = 0; j < 32; j++) {
    float a = fabsf(v[j]);
    finite = finite && (a <= 3.402823466e38f);
    M = fmaxf(M, a);
  }
#pragma unroll
  for (int w = 0; w < 4; w++)
#pragma unroll
    for (int p = 0; p < 2; p++)
#pragma unroll
      for (int l = 0; l < 4; l++) L.r[w][p][l] = 0u;
  if (!finite || M == 0.f) {
#pragma unroll
    for (int l = 0; l < 4; l++) {
      L.off[l] = 0;
      L.kf[l] = 0.f;
    }
    return finite;
  }
  int e;
  frexpf(M, &e);            // M < 2^e
  int q = 30 - e;           // M 2^q in [2^29, 2^30)
  if (q > 126) q = 126;     // keep 2^-q a normal float (only for |x| < 2^-96)
  int sum[4] = {0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 32; j++) {
    int xi = __float2int_rn(ldexpf(v[j], q));
    int l0 = (int)(int8_t)(xi & 0xff);
    xi = (xi - l0) >> 8;
    int l1 = (int)(int8_t)(xi & 0xff);
    xi = (xi - l1) >> 8;
    int l2 = (int)(int8_t)(xi & 0xff);
    int l3 = (xi - l2) >> 8;
    const int w = j >> 3, p = j & 1, b = (j & 7) >> 1;
    L.r[w][p][0] |= ((uint32_t)l0 & 0xffu) << (8 * b);
    L.r[w][p][1] |= ((uint32_t)l1 & 0xffu) << (8 * b);
    L.r[w][p][2] |= ((uint32_t)l2 & 0xffu) << (8 * b);
    L.r[w][p][3] |= ((uint32_t)l3 & 0xffu) << (8 * b);
    sum[0] += l0;
    sum[1] += l1;
    sum[2] += l2;
    sum[3] += l3;
  }
#pragma unroll
  for (int l = 0; l < 4; l++) {
    L.off[l] = -8 * sum[l];
    L.kf[l] = ldexpf(1.0f, 8 * l - q);
  }
  return true;
}

// sum_j (n_j - 8) x_j over the 32 columns of one chunk, n_j the stored nibbles in wv.
__device__ __forceinline__ float chunk_dot(const uint4 wv, const Limbs& L) {
  int a0 = L.off[0], a1 = L.off[1], a2 = L.off[2], a3 = L.off[3];
  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int w = 0; w < 4; w++) {
    const uint32_t lo = words[w] & 0x0f0f0f0fu;          // even columns, one per byte
    const uint32_t hi = (words[w] >> 4) & 0x0f0f0f0fu;   // odd columns
    a0 = dp4a_us(lo, L.r[w][0][0], a0);
    a1 = dp4a_us(lo, L.r[w][0][1], a1);
    a2 = dp4a_us(lo, L.r[w][0][2], a2);
    a3 = dp4a_us(lo, L.r[w][0][3], a3);
    a0 = dp4a_us(hi, L.r[w][1][0], a0);
    a1 = dp4a_us(hi, L.r[w][1][1], a1);
    a2 = dp4a_us(hi, L.r[w][1][2], a2);
    a3 = dp4a_us(hi, L.r[w][1][3], a3);
  }
  return fmaf(__int2float_rn(a3), L.kf[3],
              fmaf(__int2float_rn(a2), L.kf[2], fmaf(__int2float_rn(a1), L.kf[1], __int2float_rn(a0) * L.kf[0])));
}

// Any even gs that is not a multiple of 32: a chunk may cross group boundaries, so each column
// takes its own group's scale (binary32 products and sums, columns in order). The activations are
// re-read from memory (act[base + col]). Returns the scaled partial sum.
__device__ __noinline__ float chunk_dot_generic(const uint4 wv, const void* act, int dtype, size_t base,
                                                const TensorDesc T, int row, int c) {
  const float* srow = T.s + (size_t)row * T.G;
  const int col0 = 32 * c;
  int g = col0 / T.gs;
  int next = (g + 1) * T.gs;
  float acc = 0.f;
  for (int j = 0; j < 32; j++) {
    const int col = col0 + j;
    if (col >= T.cols) break;
    if (col >= next) {
      g++;
      next += T.gs;
    }
    const uint32_t word = j < 8 ? wv.x : (j < 16 ? wv.y : (j < 24 ? wv.z : wv.w));
    const int n = (int)((word >> (4 * (j & 7))) & 0xfu) - 8;
    acc = fmaf(__ldg(srow + g) * (float)n, load_act(act, dtype, base + col), acc);
  }
  return acc;
}

// Butterfly reduction of N values per lane across the warp: afterwards lane l holds, in v[0],
// the warp total of value l / (32 / N). N - 1 + log2(32 / N) shuffles.
template <int N>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[N], int lane) {
#pragma unroll
  for (int cnt = N, off = 16; cnt > 1; cnt >>= 1, off >>= 1) {
    const bool upper = lane & off;
    const int half = cnt >> 1;
#pragma unroll
    for (int i = 0; i < half; i++) {
      float send = upper ? v[i] : v[i + half];
      float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (int off = 16 / N; off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ void load_chunk_f32(const void* p, int dtype, size_t base, int col0, int cols,
                                               float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; j++) v[j] = (col0 + j < cols) ? load_act(p, dtype, base + col0 + j) : 0.f;
}

__device__ __forceinline__ TensorDesc load_desc(const TensorDesc* p) {
  TensorDesc d;
  d.w = p->w;
  d.s = p->s;
  d.pitch = p->pitch;
  d.gs = p->gs;
  d.G = p->G;
  d.rows = p->rows;
  d.cols = p->cols;
  d.mode = p->mode;
  return d;
}

// ------------------------------------------------------------------------------------------
// Route plan: kept slots of all tokens, compacted. pre[t] = sum_{t' < t} kept(t').
// ------------------------------------------------------------------------------------------

__device__ int build_plan(const int32_t* __restrict__ n_sel, int S, int K, int* pre, int* scratch32) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
  int carry = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int t = base + tid;
    int v = 0;
    if (t < S) {
      v = n_sel ? __ldg(n_sel + t) : K;
      v = v < 0 ? 0 : (v > K ? K : v);
    }
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) scratch32[warp] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
    for (int i = 0; i < nw; i++) {
      int s = scratch32[i];
      if (i < warp) wbase += s;
      total += s;
    }
    if (t < S) pre[t] = carry + wbase + incl - v;
    carry += total;
    __syncthreads();
  }
  if (tid == 0) pre[S] = carry;
  __syncthreads();
  return carry;
}

__device__ __forceinline__ int route_token(const int* pre, int S, int j) {
  int lo = 0, hi = S - 1;  // largest t with pre[t] <= j
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= j) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct GroupParams {
  const void* x;
  int x_dtype;
  int S, D, I, K;
  const int32_t* idx;
  const float* w;
  const int32_t* n_sel;
  const ExpertDesc* table;
  const void* resid;
  void* y;
  float* h;        // [routes x I]
  float* yr;       // [routes x D] (S > 1)
  int* plan;       // pre[0..S] (written by CTA 0 of the gate/up kernel)
  int* err;
};

// ------------------------------------------------------------------------------------------
// Gate + up dual GEMV with SiLU(g) * u epilogue. Thread c of the CTA owns column chunk c.
// Work = kept routes x I row pairs, split into equal contiguous ranges over the grid.
// ------------------------------------------------------------------------------------------

constexpr int kGU = 4;  // row pairs per batch (8 weight rows in flight per thread)

template <int MAXT>
__global__ void __launch_bounds__(MAXT) gateup_kernel(GroupParams P) {
  extern __shared__ int smem_plan[];        // S + 1
  __shared__ int scratch32[32];
  __shared__ float red[2][32][2 * kGU];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int C = (P.D + 31) >> 5;
  const int c = tid;
  const bool has_chunk = c < C;
  const int R = build_plan(P.n_sel, P.S, P.K, smem_plan, scratch32);
  if (blockIdx.x == 0)
    for (int t = tid; t <= P.S; t += blockDim.x) P.plan[t] = smem_plan[t];
  const long long T = (long long)R * P.I;
  long long p = (long long)blockIdx.x * T / gridDim.x;
  const long long pend = (long long)(blockIdx.x + 1) * T / gridDim.x;

  Limbs L;
  float xv[32];
  int cur_tok = -1, cur_route = -1;
  bool route_ok = false;
  TensorDesc Tg, Tu;
  int buf = 0;
  while (p < pend) {
    const int j = (int)(p / P.I);
    const int i0 = (int)(p - (long long)j * P.I);
    int nb = kGU;
    if (nb > P.I - i0) nb = P.I - i0;
    if (nb > pend - p) nb = (int)(pend - p);
    if (j != cur_route) {
      cur_route = j;
      const int t = route_token(smem_plan, P.S, j);
      const int k = j - smem_plan[t];
      const int e = __ldg(P.idx + (size_t)t * P.K + k);
      route_ok = e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
      if (!route_ok) {
        if (tid == 0) set_error(P.err, COLI_E_ROUTE);
      } else {
        Tg = load_desc(&P.table[e].t[T_GATE]);
        Tu = load_desc(&P.table[e].t[T_UP]);
      }
      if (t != cur_tok) {
        cur_tok = t;
        load_chunk_f32(P.x, P.x_dtype, (size_t)t * P.D, 32 * c, has_chunk ? P.D : 0, xv);
        if (!make_limbs(xv, L)) set_error(P.err, COLI_E_NONFINITE);
      }
    }
    float part[2 * kGU];
    if (route_ok && has_chunk) {
      uint4 wv[2 * kGU];
#pragma unroll
      for (int u = 0; u < kGU; u++) {
        if (u < nb) {
          wv[u] = ldg_stream(Tg.w + (size_t)(i0 + u) * Tg.pitch + 16 * c);
          wv[kGU + u] = ldg_stream(Tu.w + (size_t)(i0 + u) * Tu.pitch + 16 * c);
        } else {
          wv[u] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
          wv[kGU + u] = wv[u];
        }
      }
#pragma unroll
      for (int u = 0; u < 2 * kGU; u++) {
        const TensorDesc& T = u < kGU ? Tg : Tu;
        const int row = i0 + (u % kGU);
        float d;
        if (T.mode == SCALE_GENERIC) {
          d = (u % kGU) < nb ? chunk_dot_generic(wv[u], P.x, P.x_dtype, (size_t)cur_tok * P.D, T, row, c) : 0.f;
        } else {
          d = chunk_dot(wv[u], L);
          if (T.mode == SCALE_CHUNK && (u % kGU) < nb) d *= __ldg(T.s + (size_t)row * T.G + (32 * c) / T.gs);
        }
        part[u] = d;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 2 * kGU; u++) part[u] = 0.f;
    }
    warp_transpose_reduce<2 * kGU>(part, lane);
    if ((lane & (32 / (2 * kGU) - 1)) == 0) red[buf][warp][lane / (32 / (2 * kGU))] = part[0];
    __syncthreads();
    if (tid < nb && route_ok) {
      float g = 0.f, uu = 0.f;
      for (int wi = 0; wi < nwarps; wi++) {
        g += red[buf][wi][tid];
        uu += red[buf][wi][kGU + tid];
      }
      const int i = i0 + tid;
      if (Tg.mode == SCALE_ROW) g *= __ldg(Tg.s + i);
      if (Tu.mode == SCALE_ROW) uu *= __ldg(Tu.s + i);
      P.h[(size_t)j * P.I + i] = silu_mul(g, uu);
    }
    buf ^= 1;
    p += nb;
  }
}

// ------------------------------------------------------------------------------------------
// S == 1: down GEMV of every kept slot, weighting and the slot-ordered reduce in one kernel.
// Threads (k, c): slot k = tid / TPE owns column chunk c = tid % TPE of its expert's down rows.
// ------------------------------------------------------------------------------------------

constexpr int kDU = 4;  // down rows per batch

template <int MAXT>
__global__ void __launch_bounds__(MAXT) down_fused_kernel(GroupParams P, int TPE) {
  __shared__ float red[2][32][kDU];
  __shared__ float wk_s[COLI_MAX_K];
  __shared__ const float* srow_s[COLI_MAX_K];   // per-row scales of slot k (ROW mode) or null
  __shared__ int ok_s[COLI_MAX_K];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = tid / TPE, c = tid % TPE;
  const int CI = (P.I + 31) >> 5;
  int m = P.n_sel ? __ldg(P.n_sel) : P.K;
  m = m < 0 ? 0 : (m > P.K ? P.K : m);
  const int wpe = TPE >> 5;  // warps per slot
  bool active = k < m && c < CI;
  TensorDesc Td;
  int e = -1;
  if (k < m) {
    e = __ldg(P.idx + k);
    if (e < 0 || e >= COLI_MAX_EXPERTS || !P.table[e].valid) {
      e = -1;
      active = false;
    } else {
      Td = load_desc(&P.table[e].t[T_DOWN]);
    }
  }
  if (c == 0 && k < P.K) {
    ok_s[k] = (k < m && e >= 0);
    wk_s[k] = k < m ? __ldg(P.w + k) : 0.f;
    srow_s[k] = (e >= 0 && Td.mode == SCALE_ROW) ? Td.s : nullptr;
    if (k < m && e < 0) set_error(P.err, COLI_E_ROUTE);
  }
  float hv[32];
  Limbs L;
  load_chunk_f32(P.h, COLI_DTYPE_F32, (size_t)k * P.I, 32 * c, active ? P.I : 0, hv);
  if (!make_limbs(hv, L)) set_error(P.err, COLI_E_NONFINITE);
  __syncthreads();

  const int d_begin = (int)((long long)blockIdx.x * P.D / gridDim.x);
  const int d_end = (int)((long long)(blockIdx.x + 1) * P.D / gridDim.x);
  int buf = 0;
  for (int d0 = d_begin; d0 < d_end; d0 += kDU) {
    const int nb = min(kDU, d_end - d0);
    float part[kDU];
    if (active) {
      uint4 wv[kDU];
#pragma unroll
      for (int u = 0; u < kDU; u++)
        wv[u] = u < nb ? ldg_stream(Td.w + (size_t)(d0 + u) * Td.pitch + 16 * c)
                       : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
#pragma unroll
      for (int u = 0; u < kDU; u++) {
        float d;
        if (Td.mode == SCALE_GENERIC) {
          d = u < nb ? chunk_dot_generic(wv[u], P.h, COLI_DTYPE_F32, (size_t)k * P.I, Td, d0 + u, c) : 0.f;
        } else {
          d = chunk_dot(wv[u], L);
          if (Td.mode == SCALE_CHUNK && u < nb) d *= __ldg(Td.s + (size_t)(d0 + u) * Td.G + (32 * c) / Td.gs);
        }
        part[u] = d;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kDU; u++) part[u] = 0.f;
    }
    warp_transpose_reduce<kDU>(part, lane);
    if ((lane & (32 / kDU - 1)) == 0) red[buf][warp][lane / (32 / kDU)] = part[0];
    __syncthreads();
    if (tid < nb) {
      const int d = d0 + tid;
      float acc = 0.f;
      for (int kk = 0; kk < m; kk++) {
        if (!ok_s[kk]) continue;
        float yk = 0.f;
        for (int wi = kk * wpe; wi < (kk + 1) * wpe; wi++) yk += red[buf][wi][tid];
        if (srow_s[kk]) yk *= __ldg(srow_s[kk] + d);
        acc = fmaf(wk_s[kk], yk, acc);
      }
      if (P.resid) acc = load_act(P.resid, P.x_dtype, d) + acc;
      if (P.x_dtype == COLI_DTYPE_F32)
        static_cast<float*>(P.y)[d] = acc;
      else
        static_cast<uint16_t*>(P.y)[d] = f32_to_bf16_rn(acc);
    }
    buf ^= 1;
  }
}

// ------------------------------------------------------------------------------------------
// S > 1: down GEMV per kept route into yr, then a slot-ordered combine per token.
// ------------------------------------------------------------------------------------------

template <int MAXT>
__global__ void __launch_bounds__(MAXT) down_routes_kernel(GroupParams P) {
  __shared__ float red[2][32][kDU];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int CI = (P.I + 31) >> 5;
  const int c = tid;
  const bool has_chunk = c < CI;
  const int R = P.plan[P.S];
  const long long T = (long long)R * P.D;
  long long p = (long long)blockIdx.x * T / gridDim.x;
  const long long pend = (long long)(blockIdx.x + 1) * T / gridDim.x;
  Limbs L;
  float hv[32];
  int cur_route = -1;
  bool route_ok = false;
  TensorDesc Td;
  int buf = 0;
  while (p < pend) {
    const int j = (int)(p / P.D);
    const int d0 = (int)(p - (long long)j * P.D);
    int nb = kDU;
    if (nb > P.D - d0) nb = P.D - d0;
    if (nb > pend - p) nb = (int)(pend - p);
    if (j != cur_route) {
      cur_route = j;
      // route j -> token t, slot k (plan written by the gate/up kernel)
      int lo = 0, hi = P.S - 1;
      while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.plan[mid] <= j) lo = mid; else hi = mid - 1;
      }
      const int t = lo, k = j - P.plan[t];
      const int e = __ldg(P.idx + (size_t)t * P.K + k);
      route_ok = e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
      if (route_ok) Td = load_desc(&P.table[e].t[T_DOWN]);
      load_chunk_f32(P.h, COLI_DTYPE_F32, (size_t)j * P.I, 32 * c, (has_chunk && route_ok) ? P.I : 0, hv);
      if (!make_limbs(hv, L)) set_error(P.err, COLI_E_NONFINITE);
    }
    float part[kDU];
    if (route_ok && has_chunk) {
      uint4 wv[kDU];
#pragma unroll
      for (int u = 0; u < kDU; u++)
        wv[u] = u < nb ? ldg_stream(Td.w + (size_t)(d0 + u) * Td.pitch + 16 * c)
                       : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
#pragma unroll
      for (int u = 0; u < kDU; u++) {
        float d;
        if (Td.mode == SCALE_GENERIC) {
          d = u < nb ? chunk_dot_generic(wv[u], P.h, COLI_DTYPE_F32, (size_t)j * P.I, Td, d0 + u, c) : 0.f;
        } else {
          d = chunk_dot(wv[u], L);
          if (Td.mode == SCALE_CHUNK && u < nb) d *= __ldg(Td.s + (size_t)(d0 + u) * Td.G + (32 * c) / Td.gs);
        }
        part[u] = d;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kDU; u++) part[u] = 0.f;
    }
    warp_transpose_reduce<kDU>(part, lane);
    if ((lane & (32 / kDU - 1)) == 0) red[buf][warp][lane / (32 / kDU)] = part[0];
    __syncthreads();
    if (tid < nb) {
      float yk = 0.f;
      for (int wi = 0; wi < nwarps; wi++) yk += red[buf][wi][tid];
      if (route_ok && Td.mode == SCALE_ROW) yk *= __ldg(Td.s + d0 + tid);
      P.yr[(size_t)j * P.D + d0 + tid] = route_ok ? yk : 0.f;
    }
    buf ^= 1;
    p += nb;
  }
}

__global__ void combine_kernel(GroupParams P) {
  const long long n = (long long)P.S * P.D;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / P.D), d = (int)(i - (long long)t * P.D);
    const int j0 = P.plan[t], m = P.plan[t + 1] - j0;
    float acc = 0.f;
    for (int k = 0; k < m; k++) acc = fmaf(__ldg(P.w + (size_t)t * P.K + k), P.yr[(size_t)(j0 + k) * P.D + d], acc);
    if (P.resid) acc = load_act(P.resid, P.x_dtype, i) + acc;
    if (P.x_dtype == COLI_DTYPE_F32)
      static_cast<float*>(P.y)[i] = acc;
    else
      static_cast<uint16_t*>(P.y)[i] = f32_to_bf16_rn(acc);
  }
}

// ------------------------------------------------------------------------------------------
// Host launcher
// ------------------------------------------------------------------------------------------


int launch_expert_group(coli_ctx* ctx, const void* x, int x_dtype, int S, const int32_t* idx, const float* w,
                        const int32_t* n_sel, int K, const void* resid, void* y) {
  if (S > COLI_MAX_GROUP_TOKENS) return fail(ctx, COLI_E_INVAL, "expert_group: S above COLI_MAX_GROUP_TOKENS");
  const int D = ctx->table_D, I = ctx->table_I;
  const size_t R = (size_t)S * K;
  const size_t h_bytes = align_up(R * I * sizeof(float), 256);
  const size_t yr_bytes = S > 1 ? align_up(R * D * sizeof(float), 256) : 0;
  const size_t plan_bytes = align_up((size_t)(S + 1) * sizeof(int), 256);
  int rc = ensure_workspace(ctx, h_bytes + yr_bytes + plan_bytes);
  if (rc != COLI_OK) return rc;
  GroupParams P;
  P.x = x;
  P.x_dtype = x_dtype;
  P.S = S;
  P.D = D;
  P.I = I;
  P.K = K;
  P.idx = idx;
  P.w = w;
  P.n_sel = n_sel;
  P.table = ctx->d_table;
  P.resid = resid;
  P.y = y;
  P.h = reinterpret_cast<float*>(ctx->ws.base);
  P.yr = reinterpret_cast<float*>(ctx->ws.base + h_bytes);
  P.plan = reinterpret_cast<int*>(ctx->ws.base + h_bytes + yr_bytes);
  P.err = ctx->d_status;

  const int CD = (D + 31) / 32, CI = (I + 31) / 32;
  const int nt_gu = (CD + 31) / 32 * 32;
  const size_t smem_gu = (size_t)(S + 1) * sizeof(int);
  cudaError_t e;
  {
    auto kern = nt_gu <= 256 ? gateup_kernel<256> : (nt_gu <= 512 ? gateup_kernel<512> : gateup_kernel<1024>);
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nt_gu, smem_gu);
    ProfScope prof(ctx, COLI_KERNEL_GATEUP);
    kern<<<ctx->num_sms * (occ > 0 ? occ : 1), nt_gu, smem_gu, ctx->stream>>>(P);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "gate/up launch");
  }
  const int TPE = (CI + 31) / 32 * 32;
  if (S == 1 && K * TPE <= 1024) {
    const int nt = K * TPE;
    auto kern = nt <= 256 ? down_fused_kernel<256> : (nt <= 512 ? down_fused_kernel<512> : down_fused_kernel<1024>);
    int grid = ctx->num_sms;
    if (grid > D) grid = D;
    ProfScope prof(ctx, COLI_KERNEL_DOWN);
    kern<<<grid, nt, 0, ctx->stream>>>(P, TPE);
  } else {
    auto kern = TPE <= 256 ? down_routes_kernel<256> : (TPE <= 512 ? down_routes_kernel<512> : down_routes_kernel<1024>);
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, TPE, 0);
    {
      ProfScope prof(ctx, COLI_KERNEL_DOWN);
      kern<<<ctx->num_sms * (occ > 0 ? occ : 1), TPE, 0, ctx->stream>>>(P);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "down launch");
    long long n = (long long)S * D;
    int grid = (int)((n + 255) / 256);
    if (grid > 4 * ctx->num_sms) grid = 4 * ctx->num_sms;
    ProfScope prof(ctx, COLI_KERNEL_COMBINE);
    combine_kernel<<<grid, 256, 0, ctx->stream>>>(P);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "down/combine launch");
  return COLI_OK;
}

}  // namespace coli
