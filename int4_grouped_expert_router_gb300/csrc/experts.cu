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
#include "pipe.h"

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
      v = n_sel ? ld_cg_i32(n_sel + t) : K;
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
// Batches of the gate/up work: kept routes x I row pairs, split into equal contiguous ranges over
// the grid; a batch is up to RB consecutive row pairs of one route. Producer and consumers walk
// the same sequence.
// ------------------------------------------------------------------------------------------

struct RouteInfo {
  int j = -1, t = -1, k = 0, e = -1;
  bool ok = false;
};

__device__ __forceinline__ void resolve_route(const GroupParams& P, const int* pre, int j, RouteInfo& r) {
  r.j = j;
  r.t = route_token(pre, P.S, j);
  r.k = j - pre[r.t];
  r.e = ld_cg_i32(P.idx + (size_t)r.t * P.K + r.k);
  r.ok = r.e >= 0 && r.e < COLI_MAX_EXPERTS && P.table[r.e].valid;
}

// ------------------------------------------------------------------------------------------
// Gate + up dual GEMV with the SiLU(g) * u epilogue (warp-specialised, TMA-fed).
// Warps 0..W-1 are consumers: thread c owns column chunk c of every row and keeps that chunk of
// the activation in registers. Warp W is the producer: one lane streams each batch's gate and up
// rows (contiguous in memory) into a ring of NST shared-memory stages with bulk copies.
// ------------------------------------------------------------------------------------------

constexpr int kMaxStages = 8;

template <int RB>
struct GateUpSmem {
  static constexpr int kRows = 2 * RB;
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  float red[2][32][kRows];
  int abort_flag;
};

template <int RB, int MAXT>
__global__ void __launch_bounds__(MAXT) gateup_kernel(GroupParams P, uint32_t pitch, uint32_t NST) {
  using SM = GateUpSmem<RB>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t stage_bytes = 2u * RB * pitch;
  uint8_t* stages = smem_raw;
  SM& sm = *reinterpret_cast<SM*>(smem_raw + (size_t)NST * stage_bytes);
  int* pre = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(&sm) + sizeof(SM));
  __shared__ int scratch32[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = (P.D + 31) >> 5;
  const int W = (C + 31) >> 5;            // consumer warps
  const bool producer = warp == W;
  const int c = tid;
  const bool has_chunk = !producer && c < C;

  if (tid == 0) {
    for (int s = 0; s < NST; s++) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], W);
    }
    sm.abort_flag = 0;
    mbar_fence_init();
  }
  // prologue overlapping the router's tail: activation limbs of token 0
  Limbs L;
  float xv[32];
  int cur_tok = 0;
  load_chunk_f32(P.x, P.x_dtype, 0, 32 * c, has_chunk ? P.D : 0, xv);
  bool finite = make_limbs(xv, L);
  griddep_wait();
  const int R = build_plan(P.n_sel, P.S, P.K, pre, scratch32);  // contains __syncthreads
  if (blockIdx.x == 0)
    for (int t = tid; t <= P.S; t += blockDim.x) P.plan[t] = pre[t];
  griddep_launch_dependents();
  if (!finite && has_chunk) set_error(P.err, COLI_E_NONFINITE);

  const long long T = (long long)R * P.I;
  const long long pbeg = (long long)blockIdx.x * T / gridDim.x;
  const long long pend = (long long)(blockIdx.x + 1) * T / gridDim.x;

  if (producer) {
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      RouteInfo r;
      const uint8_t *wg = nullptr, *wu = nullptr;
      uint32_t b = 0;
      bool aborted = false;
      for (long long p = pbeg; p < pend && !aborted;) {
        const int j = (int)(p / P.I), i0 = (int)(p - (long long)j * P.I);
        const int nb = (int)min((long long)min(RB, P.I - i0), pend - p);
        p += nb;
        if (j != r.j) {
          resolve_route(P, pre, j, r);
          if (r.ok) {
            wg = P.table[r.e].t[T_GATE].w;
            wu = P.table[r.e].t[T_UP].w;
          }
        }
        if (!r.ok) continue;
        const uint32_t slot = b % NST;
        if (b >= NST) {
          const uint32_t par = ((b / NST) - 1) & 1;
          uint32_t spins = 0;
          while (!mbar_test_parity(&sm.empty[slot], par)) {
            if (++spins > kSpinLimit || *(volatile int*)&sm.abort_flag) {
              aborted = true;
              break;
            }
          }
          if (aborted) break;
        }
        uint8_t* st = stages + (size_t)slot * stage_bytes;
        mbar_arrive_expect_tx(&sm.full[slot], 2u * nb * pitch);
        bulk_g2s_stream(st, wg + (size_t)i0 * pitch, nb * pitch, &sm.full[slot], policy);
        bulk_g2s_stream(st + (size_t)RB * pitch, wu + (size_t)i0 * pitch, nb * pitch, &sm.full[slot], policy);
        b++;
      }
      if (aborted) set_error(P.err, COLI_E_TIMEOUT);
      // never leave the CTA with bulk copies in flight: wait for the last fill of every slot
      for (uint32_t q = b > NST ? b - NST : 0; q < b; q++) (void)mbar_wait(&sm.full[q % NST], (q / NST) & 1);
    }
    return;
  }

  // ---------------- consumers ----------------
  RouteInfo r;
  TensorDesc Tg, Tu;
  uint32_t b = 0;
  int buf = 0;
  for (long long p = pbeg; p < pend;) {
    const int j = (int)(p / P.I), i0 = (int)(p - (long long)j * P.I);
    const int nb = (int)min((long long)min(RB, P.I - i0), pend - p);
    p += nb;
    if (j != r.j) {
      resolve_route(P, pre, j, r);
      if (r.ok) {
        Tg = load_desc(&P.table[r.e].t[T_GATE]);
        Tu = load_desc(&P.table[r.e].t[T_UP]);
        if (r.t != cur_tok) {
          cur_tok = r.t;
          load_chunk_f32(P.x, P.x_dtype, (size_t)cur_tok * P.D, 32 * c, has_chunk ? P.D : 0, xv);
          if (!make_limbs(xv, L) && has_chunk) set_error(P.err, COLI_E_NONFINITE);
        }
      } else if (tid == 0) {
        set_error(P.err, COLI_E_ROUTE);
      }
    }
    if (!r.ok) continue;
    // scales needed after the wait, fetched before it
    float scg[RB], scu[RB];
#pragma unroll
    for (int u = 0; u < RB; u++) {
      scg[u] = 1.f;
      scu[u] = 1.f;
      if (u < nb && has_chunk) {
        if (Tg.mode == SCALE_CHUNK) scg[u] = __ldg(Tg.s + (size_t)(i0 + u) * Tg.G + (32 * c) / Tg.gs);
        if (Tu.mode == SCALE_CHUNK) scu[u] = __ldg(Tu.s + (size_t)(i0 + u) * Tu.G + (32 * c) / Tu.gs);
      }
    }
    float fg = 1.f, fu = 1.f;
    if (tid < nb) {
      if (Tg.mode == SCALE_ROW) fg = __ldg(Tg.s + i0 + tid);
      if (Tu.mode == SCALE_ROW) fu = __ldg(Tu.s + i0 + tid);
    }
    const uint32_t slot = b % NST;
    const bool ok = mbar_wait(&sm.full[slot], (b / NST) & 1);
    const uint8_t* st = stages + (size_t)slot * stage_bytes;
    float part[2 * RB];
#pragma unroll
    for (int u = 0; u < 2 * RB; u++) {
      const int uu = u % RB;
      const TensorDesc& T = u < RB ? Tg : Tu;
      float d = 0.f;
      if (ok && has_chunk && uu < nb) {
        const uint4 wv = lds128(st + (size_t)(u < RB ? 0 : RB) * pitch + (size_t)uu * pitch + 16 * c);
        if (T.mode == SCALE_GENERIC)
          d = chunk_dot_generic(wv, P.x, P.x_dtype, (size_t)cur_tok * P.D, T, i0 + uu, c);
        else
          d = chunk_dot(wv, L) * (u < RB ? scg[uu] : scu[uu]);
      }
      part[u] = d;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);
    warp_transpose_reduce<2 * RB>(part, lane);
    if ((lane & (32 / (2 * RB) - 1)) == 0) sm.red[buf][warp][lane / (32 / (2 * RB))] = part[0];
    if (named_sync_or(1, W * 32, !ok)) {  // uniform decision across the consumer warps
      if (tid == 0) {
        set_error(P.err, COLI_E_TIMEOUT);
        *(volatile int*)&sm.abort_flag = 1;
      }
      break;
    }
    if (tid < nb) {
      float g = 0.f, u = 0.f;
      for (int wi = 0; wi < W; wi++) {
        g += sm.red[buf][wi][tid];
        u += sm.red[buf][wi][RB + tid];
      }
      P.h[(size_t)j * P.I + i0 + tid] = silu_mul(g * fg, u * fu);
    }
    buf ^= 1;
    b++;
  }
}

// ------------------------------------------------------------------------------------------
// S == 1: down GEMV of every kept slot, weighting and the slot-ordered reduce in one kernel
// (warp-specialised, TMA-fed). Consumer threads (k, c): slot k = tid / TPE owns column chunk
// c = tid % TPE of its expert's down rows, with that chunk of h_k in registers. The producer warp
// streams, per batch of RB output rows, the RB rows of every kept expert (one bulk copy each).
// The weight stream does not depend on the gate/up kernel, so it starts before that kernel ends.
// ------------------------------------------------------------------------------------------

template <int RB>
struct DownSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  float red[2][32][RB];
  float rscale[2][COLI_MAX_K][RB];
  float wk[COLI_MAX_K];
  int ok[COLI_MAX_K];
  int mode_row[COLI_MAX_K];
  int abort_flag;
};

template <int RB, int MAXT>
__global__ void __launch_bounds__(MAXT) down_fused_kernel(GroupParams P, int TPE, uint32_t pitch, uint32_t NST) {
  using SM = DownSmem<RB>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t slot_bytes = (uint32_t)P.K * RB * pitch;  // per stage: K experts x RB rows
  uint8_t* stages = smem_raw;
  SM& sm = *reinterpret_cast<SM*>(smem_raw + (size_t)NST * slot_bytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = P.K * TPE;               // consumer threads
  const int WC = NC >> 5;
  const bool producer = tid >= NC;
  const int k = tid / TPE, c = tid % TPE;
  const int CI = (P.I + 31) >> 5;
  const int wpe = TPE >> 5;

  // routes of token 0 (written by the router, complete before the gate/up kernel started)
  int m = P.n_sel ? ld_cg_i32(P.n_sel) : P.K;
  m = m < 0 ? 0 : (m > P.K ? P.K : m);
  if (tid == 0) {
    for (int s = 0; s < NST; s++) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], WC);
    }
    sm.abort_flag = 0;
    mbar_fence_init();
  }
  if (!producer && c == 0) {
    int e = k < m ? ld_cg_i32(P.idx + k) : -1;
    bool ok = k < m && e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
    if (k < m && !ok) set_error(P.err, COLI_E_ROUTE);
    sm.ok[k] = ok;
    sm.wk[k] = ok ? ld_cg_f32(P.w + k) : 0.f;
    sm.mode_row[k] = ok ? (P.table[e].t[T_DOWN].mode == SCALE_ROW) : 0;
  }
  __syncthreads();
  const int d_begin = (int)((long long)blockIdx.x * P.D / gridDim.x);
  const int d_end = (int)((long long)(blockIdx.x + 1) * P.D / gridDim.x);

  if (producer) {
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      const uint8_t* wsrc[COLI_MAX_K];
      for (int kk = 0; kk < m; kk++) wsrc[kk] = sm.ok[kk] ? P.table[ld_cg_i32(P.idx + kk)].t[T_DOWN].w : nullptr;
      uint32_t b = 0;
      bool aborted = false;
      for (int d0 = d_begin; d0 < d_end; d0 += RB, b++) {
        const int nb = min(RB, d_end - d0);
        const uint32_t slot = b % NST;
        if (b >= NST) {
          const uint32_t par = ((b / NST) - 1) & 1;
          uint32_t spins = 0;
          while (!mbar_test_parity(&sm.empty[slot], par)) {
            if (++spins > kSpinLimit || *(volatile int*)&sm.abort_flag) {
              aborted = true;
              break;
            }
          }
          if (aborted) break;
        }
        uint32_t bytes = 0;
        for (int kk = 0; kk < m; kk++)
          if (wsrc[kk]) bytes += nb * pitch;
        uint8_t* st = stages + (size_t)slot * slot_bytes;
        mbar_arrive_expect_tx(&sm.full[slot], bytes);
        for (int kk = 0; kk < m; kk++)
          if (wsrc[kk])
            bulk_g2s_stream(st + (size_t)kk * RB * pitch, wsrc[kk] + (size_t)d0 * pitch, nb * pitch, &sm.full[slot],
                            policy);
      }
      if (aborted) set_error(P.err, COLI_E_TIMEOUT);
      for (uint32_t q = b > NST ? b - NST : 0; q < b; q++) (void)mbar_wait(&sm.full[q % NST], (q / NST) & 1);
    }
    return;
  }

  // ---------------- consumers ----------------
  const bool active = k < m && sm.ok[k] && c < CI;
  TensorDesc Td;
  if (active) Td = load_desc(&P.table[ld_cg_i32(P.idx + k)].t[T_DOWN]);
  griddep_wait();  // h is written by the gate/up kernel
  float hv[32];
  Limbs L;
  load_chunk_f32(P.h, COLI_DTYPE_F32, (size_t)k * P.I, 32 * c, active ? P.I : 0, hv);
  if (!make_limbs(hv, L) && active) set_error(P.err, COLI_E_NONFINITE);

  uint32_t b = 0;
  int buf = 0;
  for (int d0 = d_begin; d0 < d_end; d0 += RB, b++) {
    const int nb = min(RB, d_end - d0);
    float sc[RB];
    float rs[RB];
#pragma unroll
    for (int u = 0; u < RB; u++) {
      sc[u] = 1.f;
      rs[u] = 1.f;
      if (active && u < nb) {
        if (Td.mode == SCALE_CHUNK) sc[u] = __ldg(Td.s + (size_t)(d0 + u) * Td.G + (32 * c) / Td.gs);
        if (Td.mode == SCALE_ROW && c == 0) rs[u] = __ldg(Td.s + d0 + u);
      }
    }
    float res = 0.f;
    if (tid < nb && P.resid) res = load_act(P.resid, P.x_dtype, d0 + tid);
    const uint32_t slot = b % NST;
    const bool ok = mbar_wait(&sm.full[slot], (b / NST) & 1);
    const uint8_t* st = stages + (size_t)slot * slot_bytes + (size_t)k * RB * pitch;
    float part[RB];
#pragma unroll
    for (int u = 0; u < RB; u++) {
      float d = 0.f;
      if (ok && active && u < nb) {
        const uint4 wv = lds128(st + (size_t)u * pitch + 16 * c);
        if (Td.mode == SCALE_GENERIC)
          d = chunk_dot_generic(wv, P.h, COLI_DTYPE_F32, (size_t)k * P.I, Td, d0 + u, c);
        else
          d = chunk_dot(wv, L) * sc[u];
      }
      part[u] = d;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);
    if (c == 0 && k < m) {
#pragma unroll
      for (int u = 0; u < RB; u++) sm.rscale[buf][k][u] = rs[u];
    }
    warp_transpose_reduce<RB>(part, lane);
    if ((lane & (32 / RB - 1)) == 0) sm.red[buf][warp][lane / (32 / RB)] = part[0];
    if (named_sync_or(1, NC, !ok)) {
      if (tid == 0) {
        set_error(P.err, COLI_E_TIMEOUT);
        *(volatile int*)&sm.abort_flag = 1;
      }
      break;
    }
    if (tid < nb) {
      const int d = d0 + tid;
      float acc = 0.f;
      for (int kk = 0; kk < m; kk++) {
        if (!sm.ok[kk]) continue;
        float yk = 0.f;
        for (int wi = kk * wpe; wi < (kk + 1) * wpe; wi++) yk += sm.red[buf][wi][tid];
        if (sm.mode_row[kk]) yk *= sm.rscale[buf][kk][tid];
        acc = fmaf(sm.wk[kk], yk, acc);
      }
      if (P.resid) acc = res + acc;
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

constexpr int kDU = 4;  // rows per batch of the route-parallel down kernel

// ------------------------------------------------------------------------------------------
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


constexpr int kGateUpRows = 2;            // row pairs per gate/up stage
constexpr int kDownRows = 2;              // output rows per down stage
constexpr uint32_t kStageBudget = 96 * 1024;  // shared memory for the stage ring of one CTA

// Launch with programmatic stream serialisation (the kernel may start while its predecessor in
// the stream finishes; it calls griddepcontrol.wait before reading that predecessor's output).
template <typename... KArgs, typename... Args>
static cudaError_t launch_k(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t st, bool pdl,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

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
  const uint32_t pitch_d = (uint32_t)CD * 16, pitch_i = (uint32_t)CI * 16;
  cudaError_t e;
  {
    constexpr int RB = kGateUpRows;
    const int nt = ((CD + 31) / 32 + 1) * 32;  // consumer warps + producer warp
    const uint32_t stage = 2u * RB * pitch_d;
    uint32_t nst = kStageBudget / stage;
    nst = nst < 2 ? 2 : (nst > kMaxStages ? kMaxStages : nst);
    const size_t smem = (size_t)nst * stage + sizeof(GateUpSmem<RB>) + (size_t)(S + 1) * sizeof(int);
    auto kern = nt <= 256 ? gateup_kernel<RB, 256> : (nt <= 512 ? gateup_kernel<RB, 512> : gateup_kernel<RB, 1024>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "gate/up smem attribute");
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nt, smem);
    ProfScope prof(ctx, COLI_KERNEL_GATEUP);
    e = launch_k(kern, ctx->num_sms * (occ > 0 ? occ : 1), nt, smem, ctx->stream, true, P, pitch_d, nst);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "gate/up launch");
  }
  const int TPE = (CI + 31) / 32 * 32;
  constexpr int RBD = kDownRows;
  const uint32_t down_stage = (uint32_t)K * RBD * pitch_i;
  if (S == 1 && K * TPE + 32 <= 1024 && 2 * down_stage <= 2 * kStageBudget) {
    const int nt = K * TPE + 32;
    uint32_t nst = kStageBudget / down_stage;
    nst = nst < 2 ? 2 : (nst > kMaxStages ? kMaxStages : nst);
    const size_t smem = (size_t)nst * down_stage + sizeof(DownSmem<RBD>);
    auto kern = nt <= 256 ? down_fused_kernel<RBD, 256>
                          : (nt <= 544 ? down_fused_kernel<RBD, 544> : down_fused_kernel<RBD, 1024>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "down smem attribute");
    int grid = ctx->num_sms;
    if (grid > D) grid = D;
    ProfScope prof(ctx, COLI_KERNEL_DOWN);
    e = launch_k(kern, grid, nt, smem, ctx->stream, true, P, TPE, pitch_i, nst);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "down launch");
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
