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

// Exact int -> float for |a| < 2^22 with an integer add and a float subtract (both on the fast
// pipes): the integer is placed in the mantissa of 1.5 * 2^23.
__device__ __forceinline__ float exact_i2f(int a) { return __int_as_float(a + 0x4B400000) - 12582912.0f; }

// sum_j (n_j - 8) x_j over the 32 columns of one chunk, n_j the stored nibbles in wv. Even and odd
// columns accumulate in separate chains (8 independent dp4a chains of 4); every partial sum is an
// exact integer below 2^17 in magnitude.
__device__ __forceinline__ float chunk_dot(const uint4 wv, const Limbs& L) {
  int a0 = L.off[0], a1 = L.off[1], a2 = L.off[2], a3 = L.off[3];
  int b0 = 0, b1 = 0, b2 = 0, b3 = 0;
  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int w = 0; w < 4; w++) {
    const uint32_t lo = words[w] & 0x0f0f0f0fu;          // even columns, one per byte
    const uint32_t hi = (words[w] >> 4) & 0x0f0f0f0fu;   // odd columns
    a0 = dp4a_us(lo, L.r[w][0][0], a0);
    a1 = dp4a_us(lo, L.r[w][0][1], a1);
    a2 = dp4a_us(lo, L.r[w][0][2], a2);
    a3 = dp4a_us(lo, L.r[w][0][3], a3);
    b0 = dp4a_us(hi, L.r[w][1][0], b0);
    b1 = dp4a_us(hi, L.r[w][1][1], b1);
    b2 = dp4a_us(hi, L.r[w][1][2], b2);
    b3 = dp4a_us(hi, L.r[w][1][3], b3);
  }
  return fmaf(exact_i2f(a3 + b3), L.kf[3],
              fmaf(exact_i2f(a2 + b2), L.kf[2], fmaf(exact_i2f(a1 + b1), L.kf[1], exact_i2f(a0 + b0) * L.kf[0])));
}

// Any even gs that is not a multiple of 32: a chunk may cross group boundaries, so each column
// takes its own group's scale (binary32 products and sums, columns in order). The activations are
// re-read from memory (act[base + col]). Returns the scaled partial sum.
__device__ __noinline__ float chunk_dot_generic(const uint4 wv, const void* act, int dtype, size_t base,
                                                const TensorDesc* T, int row, int c) {
  const int gs = T->gs, G = T->G, cols = T->cols;
  const float* srow = T->s + (size_t)row * G;
  const int col0 = 32 * c;
  int g = col0 / gs;
  int next = (g + 1) * gs;
  float acc = 0.f;
  for (int j = 0; j < 32; j++) {
    const int col = col0 + j;
    if (col >= cols) break;
    if (col >= next) {
      g++;
      next += gs;
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

// v[j] = activation (f32 or bf16, widened exactly) of column col0 + j, 0 at and beyond `cols`.
// Whole chunks of aligned rows use 16-byte loads through L2.
__device__ __forceinline__ void load_chunk_f32(const void* p, int dtype, size_t base, int col0, int cols,
                                               float (&v)[32]) {
  const bool full = col0 + 32 <= cols;
  if (dtype == COLI_DTYPE_F32) {
    const float* q = static_cast<const float*>(p) + base + col0;
    if (full && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(q) + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
      return;
    }
  } else {
    const uint16_t* q = static_cast<const uint16_t*>(p) + base + col0;
    if (full && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const uint4 u = __ldcg(reinterpret_cast<const uint4*>(q) + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; h++) {
          v[8 * i + 2 * h] = __uint_as_float(w[h] << 16);
          v[8 * i + 2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
        }
      }
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < 32; j++) v[j] = (col0 + j < cols) ? load_act(p, dtype, base + col0 + j) : 0.f;
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

// ------------------------------------------------------------------------------------------
// Shared pieces of the two streaming kernels
//
// Every consumer warp owns one 512-byte column slice (32 chunks of 16 bytes) of the weight rows
// and streams it by itself: its lane 0 issues 2-D TMA loads of [kBoxRows rows x slice] boxes into
// the warp's own ring of kWarpStages shared-memory stages, kWarpStages boxes ahead of the
// warp's compute. Warps never wait for each other while streaming; they meet only at the end of a
// segment of rows to add their slices' partial sums in a fixed order.
// ------------------------------------------------------------------------------------------

constexpr int kWarpStages = 2;
constexpr int kSeg = 64;          // rows (down) or row pairs (gate/up) finished together
constexpr int kRouteCache = 16;   // routes resolved once into shared memory

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Everything a kernel needs about one tensor of a kept route, copied once into shared memory.
struct SlotTensor {
  const TensorDesc* d;  // in the device expert table (the TMA maps live there)
  const float* s;       // scales
  int mode, G, gs, box_s, box_w, box_rows;
};

struct RouteSlot {
  SlotTensor ts[2];
  int t, ok;
};

__device__ __forceinline__ void fill_slot_tensor(SlotTensor& st, const TensorDesc* d) {
  st.d = d;
  st.s = d->s;
  st.mode = d->mode;
  st.G = d->G;
  st.gs = d->gs;
  st.box_s = (int)d->box_s;
  st.box_w = (int)d->box_w;
  st.box_rows = (int)d->box_rows;
}

__device__ void resolve_slot(const GroupParams& P, const int* pre, int j, int t0, int t1, RouteSlot& rs) {
  const int t = route_token(pre, P.S, j);
  const int k = j - pre[t];
  const int e = ld_cg_i32(P.idx + (size_t)t * P.K + k);
  rs.t = t;
  rs.ok = e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
  if (rs.ok) {
    fill_slot_tensor(rs.ts[0], &P.table[e].t[t0]);
    if (t1 >= 0) fill_slot_tensor(rs.ts[1], &P.table[e].t[t1]);
  }
}

// Per-lane values for one tensor of the current route.
struct LaneTensor {
  const TensorDesc* d;
  const float* s;
  int mode, G, cg, box_s, rowB;  // cg: this lane's chunk group; rowB: bytes per box row in smem
  bool fast;                     // per-row scales, or chunk scales staged by TMA
};

__device__ __forceinline__ void lane_tensor(LaneTensor& lt, const SlotTensor& st, int c) {
  lt.d = st.d;
  lt.s = st.s;
  lt.mode = st.mode;
  lt.G = st.G;
  lt.cg = st.mode == SCALE_CHUNK ? (32 * c) / st.gs : 0;
  lt.box_s = st.box_s;
  lt.rowB = st.box_w * 4;
  lt.fast = st.mode == SCALE_ROW || (st.mode == SCALE_CHUNK && st.box_s > 0);
}

// Dot product of one staged chunk with the activation limbs, scaled by its chunk-group scale
// (per-row scales are applied after the row is complete). `sc` points at the staged scale box.
__device__ __noinline__ float chunk_dot_slow(const uint4 wv, const Limbs& L, const LaneTensor& lt, const void* act,
                                             int dtype, size_t base, int row, int c) {
  if (lt.mode == SCALE_GENERIC) return chunk_dot_generic(wv, act, dtype, base, lt.d, row, c);
  return chunk_dot(wv, L) * __ldg(lt.s + (size_t)row * lt.G + lt.cg);
}

// Walks [beg, end) over (route, row) items, `rows` rows per route, in batches of up to kBoxRows
// items that never cross a route or a segment (kSeg items from beg).
struct BatchWalk {
  int j, i, left, done, rows;
  __device__ BatchWalk(long long beg, long long end, int rows_) : rows(rows_) {
    j = (int)(beg / rows_);
    i = (int)(beg - (long long)j * rows_);
    left = (int)(end - beg);
    done = 0;
  }
  __device__ int next() const {
    int n = kBoxRows < rows - i ? kBoxRows : rows - i;
    n = n < left ? n : left;
    const int to_seg = kSeg - done % kSeg;
    return n < to_seg ? n : to_seg;
  }
  __device__ void advance(int n) {
    i += n;
    left -= n;
    done += n;
    if (i == rows) {
      i = 0;
      j++;
    }
  }
};

// ------------------------------------------------------------------------------------------
// Gate + up dual GEMV with the SiLU(g) * u epilogue.
// Thread c of the CTA owns column chunk c (warp c / 32 owns slice c / 32) of every row and keeps
// that chunk of the activation in registers. A stage of a warp holds kBoxRows gate rows and
// kBoxRows up rows of its slice (and their chunk scales when those travel by TMA).
// ------------------------------------------------------------------------------------------

struct GateUpSmem {
  RouteSlot routes[kRouteCache];
  uint64_t bars[8][kWarpStages];  // gate/up CTAs have at most 8 warps (D <= 8192)
};
// followed in dynamic shared memory by the warps' rings, pg[W][kSeg], pu[W][kSeg], pre[S + 1]

__host__ __device__ inline uint32_t gateup_stage_bytes() {
  // gate box + up box (kBoxRows x 512 B each) + two scale boxes (kBoxRows x kScaleBox floats)
  return 2u * kBoxRows * kSliceWords * 4 + 2u * kBoxRows * kScaleBox * 4;
}

inline size_t gateup_smem_bytes(int W, int S) {
  return 128 + sizeof(GateUpSmem) + (size_t)W * kWarpStages * gateup_stage_bytes() +
         2 * (size_t)W * kSeg * sizeof(float) + (size_t)(S + 1) * sizeof(int);
}

template <int MAXT>
__global__ void __launch_bounds__(MAXT, MAXT <= 192 ? 2 : 1) gateup_kernel(GroupParams P) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem_raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  const int C = (P.D + 31) >> 5;
  const int W = (C + 31) >> 5;
  const uint32_t SB = gateup_stage_bytes();
  GateUpSmem& sm = *reinterpret_cast<GateUpSmem*>(smem_raw);
  uint8_t* rings = smem_raw + sizeof(GateUpSmem);
  float* pg = reinterpret_cast<float*>(rings + (size_t)W * kWarpStages * SB);
  float* pu = pg + (size_t)W * kSeg;
  int* pre = reinterpret_cast<int*>(pu + (size_t)W * kSeg);
  __shared__ int scratch32[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid;
  const bool has_chunk = c < C;
  uint8_t* ring = rings + (size_t)warp * kWarpStages * SB;
  uint64_t* bars = sm.bars[warp];
  if (lane == 0) {
    for (int s = 0; s < kWarpStages; s++) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  // prologue overlapping the router's tail: activation limbs of token 0
  Limbs L;
  float xv[32];
  int cur_tok = 0;
  load_chunk_f32(P.x, P.x_dtype, 0, 32 * c, has_chunk ? P.D : 0, xv);
  const bool finite0 = make_limbs(xv, L);
  griddep_wait();
  const int R = build_plan(P.n_sel, P.S, P.K, pre, scratch32);  // contains __syncthreads
  if (blockIdx.x == 0)
    for (int t = tid; t <= P.S; t += blockDim.x) P.plan[t] = pre[t];
  griddep_launch_dependents();
  if (!finite0 && has_chunk) set_error(P.err, COLI_E_NONFINITE);

  const long long T = (long long)R * P.I;
  const long long pbeg = (long long)blockIdx.x * T / gridDim.x;
  const long long pend = (long long)(blockIdx.x + 1) * T / gridDim.x;
  if (pbeg >= pend) return;  // uniform across the CTA
  const int j_first = (int)(pbeg / P.I);
  const int n_routes = (int)((pend - 1) / P.I) - j_first + 1;  // <= kRouteCache (launch sizing)
  if (tid < n_routes) resolve_slot(P, pre, j_first + tid, T_GATE, T_UP, sm.routes[tid]);
  __syncthreads();

  // issue side of this warp's ring: kWarpStages batches ahead of the compute
  BatchWalk iw(pbeg, pend, P.I);
  uint32_t issued = 0;
  auto issue_next = [&]() {
    while (iw.left > 0) {
      const int n = iw.next(), j = iw.j, i0 = iw.i;
      iw.advance(n);
      const RouteSlot& rs = sm.routes[j - j_first];
      if (!rs.ok) continue;
      const uint32_t s = issued % kWarpStages;
      uint8_t* st = ring + (size_t)s * SB;
      const SlotTensor& g = rs.ts[0];
      const SlotTensor& u = rs.ts[1];
      uint32_t bytes = 2u * g.box_rows * g.box_w * 4;
      if (g.box_s) bytes += g.box_rows * g.box_s * 4;
      if (u.box_s) bytes += u.box_rows * u.box_s * 4;
      mbar_arrive_expect_tx(&bars[s], bytes);
      const int x = kSliceWords * warp;
      tma_load_2d(st, &g.d->map_w, x, i0, &bars[s]);
      tma_load_2d(st + kBoxRows * kSliceWords * 4, &u.d->map_w, x, i0, &bars[s]);
      if (g.box_s) tma_load_2d(st + 2 * kBoxRows * kSliceWords * 4, &g.d->map_s, g.box_s * warp, i0, &bars[s]);
      if (u.box_s)
        tma_load_2d(st + 2 * kBoxRows * kSliceWords * 4 + kBoxRows * kScaleBox * 4, &u.d->map_s, u.box_s * warp, i0,
                    &bars[s]);
      issued++;
      return;
    }
  };
  if (lane == 0)
    for (int s = 0; s < kWarpStages; s++) issue_next();

  // ---------------- compute ----------------
  int rj = -1;
  const RouteSlot* rs = nullptr;
  LaneTensor tg, tu;
  uint32_t b = 0;
  bool stop = false;
  int seg_n = 0;
  float fg = 1.f, fu = 1.f;  // finaliser thread `tid`: row scales of its segment row pair
  size_t hdst = 0;
  bool fin_ok = false;
  for (BatchWalk cw(pbeg, pend, P.I); cw.left > 0;) {
    const int n = cw.next(), j = cw.j, i0 = cw.i;
    cw.advance(n);
    if (j != rj) {
      rj = j;
      rs = &sm.routes[j - j_first];
      if (rs->ok) {
        lane_tensor(tg, rs->ts[0], c);
        lane_tensor(tu, rs->ts[1], c);
        if (rs->t != cur_tok) {
          cur_tok = rs->t;
          load_chunk_f32(P.x, P.x_dtype, (size_t)cur_tok * P.D, 32 * c, has_chunk ? P.D : 0, xv);
          if (!make_limbs(xv, L) && has_chunk) set_error(P.err, COLI_E_NONFINITE);
        }
      } else if (tid == 0) {
        set_error(P.err, COLI_E_ROUTE);
      }
    }
    const bool rok = rs->ok;
    if (tid >= seg_n && tid < seg_n + n) {  // finaliser of each row pair of this batch
      const int ii = i0 + (tid - seg_n);
      fin_ok = rok;
      hdst = (size_t)j * P.I + ii;
      fg = (rok && tg.mode == SCALE_ROW) ? __ldg(tg.s + ii) : 1.f;
      fu = (rok && tu.mode == SCALE_ROW) ? __ldg(tu.s + ii) : 1.f;
    }
    if (rok && !stop) {
      const uint32_t s = b % kWarpStages;
      const bool ok = mbar_wait(&bars[s], (b / kWarpStages) & 1);
      const uint8_t* st = ring + (size_t)s * SB;
      const uint8_t* sg = st + 2 * kBoxRows * kSliceWords * 4;
      const uint8_t* su = sg + kBoxRows * kScaleBox * 4;
      float acc[2 * kBoxRows];
      const int sgo = tg.cg - tg.box_s * warp, suo = tu.cg - tu.box_s * warp;  // lane's scale in the box
      if (ok && has_chunk && tg.fast && tu.fast) {
#pragma unroll
        for (int u = 0; u < kBoxRows; u++) {
          float dg = 0.f, du = 0.f;
          if (u < n) {
            dg = chunk_dot(lds128(st + u * tg.rowB + 16 * lane), L);
            du = chunk_dot(lds128(st + kBoxRows * kSliceWords * 4 + u * tu.rowB + 16 * lane), L);
            if (tg.box_s) dg *= lds32f(sg + (u * tg.box_s + sgo) * 4);
            if (tu.box_s) du *= lds32f(su + (u * tu.box_s + suo) * 4);
          }
          acc[2 * u] = dg;
          acc[2 * u + 1] = du;
        }
      } else {
        float tmp[2 * kBoxRows];  // local memory: the rarely used slow path keeps code small
#pragma unroll 1
        for (int u = 0; u < kBoxRows; u++) {
          float dg = 0.f, du = 0.f;
          if (ok && has_chunk && u < n) {
            const uint4 wg = lds128(st + u * tg.rowB + 16 * lane);
            const uint4 wu = lds128(st + kBoxRows * kSliceWords * 4 + u * tu.rowB + 16 * lane);
            const size_t xb = (size_t)cur_tok * P.D;
            dg = tg.fast ? chunk_dot(wg, L) * (tg.box_s ? lds32f(sg + (u * tg.box_s + sgo) * 4) : 1.f)
                         : chunk_dot_slow(wg, L, tg, P.x, P.x_dtype, xb, i0 + u, c);
            du = tu.fast ? chunk_dot(wu, L) * (tu.box_s ? lds32f(su + (u * tu.box_s + suo) * 4) : 1.f)
                         : chunk_dot_slow(wu, L, tu, P.x, P.x_dtype, xb, i0 + u, c);
          }
          tmp[2 * u] = dg;
          tmp[2 * u + 1] = du;
        }
#pragma unroll
        for (int v = 0; v < 2 * kBoxRows; v++) acc[v] = tmp[v];
      }
      __syncwarp();
      if (lane == 0) issue_next();  // refill the stage just consumed
      if (!ok) {
        stop = true;
        set_error(P.err, COLI_E_TIMEOUT);
      }
      // lane l ends with the warp total of value l / 2: row pair v / 2, gate (even v) or up (odd v)
      warp_transpose_reduce<2 * kBoxRows>(acc, lane);
      if ((lane & 1) == 0) {
        const int v = lane >> 1;
        if ((v >> 1) < n) ((v & 1) ? pu : pg)[warp * kSeg + seg_n + (v >> 1)] = acc[0];
      }
      b++;
    }
    seg_n += n;
    if (seg_n == kSeg || cw.left == 0) {
      const bool any_stop = named_sync_or(1, W * 32, stop);
      if (!any_stop && tid < seg_n && fin_ok) {
        float g = 0.f, u = 0.f;
        for (int wi = 0; wi < W; wi++) {
          g += pg[wi * kSeg + tid];
          u += pu[wi * kSeg + tid];
        }
        P.h[hdst] = silu_mul(g * fg, u * fu);
      }
      named_sync(1, W * 32);  // the partial buffers are reused by the next segment
      seg_n = 0;
      fin_ok = false;
      if (any_stop) stop = true;
    }
  }
  // never leave with TMA loads in flight into this warp's ring
  if (lane == 0)
    for (uint32_t q = issued > kWarpStages ? issued - kWarpStages : 0; q < issued; q++)
      if (q >= b) (void)mbar_wait(&bars[q % kWarpStages], (q / kWarpStages) & 1);
}

// ------------------------------------------------------------------------------------------
// S == 1: down GEMV of every kept slot, weighting and the slot-ordered reduce in one kernel.
// Threads (k, c): slot k = tid / TPE owns column chunk c = tid % TPE of its expert's down rows,
// with that chunk of h_k in registers; each warp streams its own slice of its expert's rows. The
// weight stream does not depend on the gate/up kernel, so it starts before that kernel ends.
// ------------------------------------------------------------------------------------------

struct DownSmem {
  uint64_t bars[32][kWarpStages];
  float part[32][kSeg];
  float rscale[COLI_MAX_K][kSeg];
  float wk[COLI_MAX_K];
  SlotTensor st[COLI_MAX_K];
  int ok[COLI_MAX_K];
};

__host__ __device__ inline uint32_t down_stage_bytes() { return kBoxRows * kSliceWords * 4 + kBoxRows * kScaleBox * 4; }

inline size_t down_smem_bytes(int nwarps) {
  return 128 + sizeof(DownSmem) + (size_t)nwarps * kWarpStages * down_stage_bytes();
}

template <int MAXT>
__global__ void __launch_bounds__(MAXT, 1) down_fused_kernel(GroupParams P, int TPE) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem_raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  DownSmem& sm = *reinterpret_cast<DownSmem*>(smem_raw);
  const uint32_t SB = down_stage_bytes();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = blockDim.x;
  const int k = tid / TPE, c = tid % TPE;
  const int CI = (P.I + 31) >> 5;
  const int wpe = TPE >> 5;
  const int slice = warp % wpe;  // this warp's column slice of its expert's rows
  uint8_t* ring = smem_raw + sizeof(DownSmem) + (size_t)warp * kWarpStages * SB;
  uint64_t* bars = sm.bars[warp];

  // routes of token 0 (written by the router, complete before the gate/up kernel started)
  int m = P.n_sel ? ld_cg_i32(P.n_sel) : P.K;
  m = m < 0 ? 0 : (m > P.K ? P.K : m);
  if (lane == 0) {
    for (int s = 0; s < kWarpStages; s++) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  if (tid < P.K) {
    bool ok = false;
    if (tid < m) {
      const int e = ld_cg_i32(P.idx + tid);
      ok = e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
      if (ok) fill_slot_tensor(sm.st[tid], &P.table[e].t[T_DOWN]);
      else set_error(P.err, COLI_E_ROUTE);
    }
    sm.ok[tid] = ok;
    sm.wk[tid] = ok ? ld_cg_f32(P.w + tid) : 0.f;
  }
  __syncthreads();
  const int d_begin = (int)((long long)blockIdx.x * P.D / gridDim.x);
  const int d_end = (int)((long long)(blockIdx.x + 1) * P.D / gridDim.x);
  const bool warp_on = k < m && sm.ok[k];  // uniform per warp
  const SlotTensor* sl = &sm.st[k < P.K ? k : 0];
  const bool active = warp_on && c < CI;

  uint32_t issued = 0;
  const uint32_t nbat = (uint32_t)((d_end - d_begin + kBoxRows - 1) / kBoxRows);
  auto issue_next = [&]() {
    if (issued >= nbat) return;
    const uint32_t s = issued % kWarpStages;
    uint8_t* st = ring + (size_t)s * SB;
    const int d0 = d_begin + (int)issued * kBoxRows;
    uint32_t bytes = sl->box_rows * sl->box_w * 4 + (sl->box_s ? sl->box_rows * sl->box_s * 4 : 0);
    mbar_arrive_expect_tx(&bars[s], bytes);
    tma_load_2d(st, &sl->d->map_w, kSliceWords * slice, d0, &bars[s]);
    if (sl->box_s) tma_load_2d(st + kBoxRows * kSliceWords * 4, &sl->d->map_s, sl->box_s * slice, d0, &bars[s]);
    issued++;
  };
  if (warp_on && lane == 0)
    for (int s = 0; s < kWarpStages; s++) issue_next();  // the weight stream starts before h is ready

  LaneTensor lt;
  lane_tensor(lt, *sl, c);
  const int so = lt.cg - lt.box_s * slice;  // lane's scale within the staged box
  griddep_wait();  // h is written by the gate/up kernel
  float hv[32];
  Limbs L;
  load_chunk_f32(P.h, COLI_DTYPE_F32, (size_t)k * P.I, 32 * c, active ? P.I : 0, hv);
  if (!make_limbs(hv, L) && active) set_error(P.err, COLI_E_NONFINITE);

  uint32_t b = 0;
  bool stop = false;
  for (int s0 = d_begin; s0 < d_end; s0 += kSeg) {
    const int nseg = min(kSeg, d_end - s0);
    // per-row scales (gs = 0) of every slot and the residual, loaded now, stored after the batches
    float rsv = 1.f;
    int rsk = -1, rsr = 0;
    if (tid < P.K * nseg) {
      rsk = tid / nseg;
      rsr = tid - rsk * nseg;
      if (rsk < m && sm.ok[rsk] && sm.st[rsk].mode == SCALE_ROW) rsv = __ldg(sm.st[rsk].s + s0 + rsr);
    }
    float res = 0.f;
    if (tid < nseg && P.resid) res = load_act(P.resid, P.x_dtype, s0 + tid);
    for (int d0 = s0; d0 < s0 + nseg; d0 += kBoxRows) {
      const int n = min(kBoxRows, s0 + nseg - d0);
      if (!warp_on || stop) continue;
      const uint32_t s = b % kWarpStages;
      const bool ok = mbar_wait(&bars[s], (b / kWarpStages) & 1);
      const uint8_t* st = ring + (size_t)s * SB;
      float acc[kBoxRows];
      if (ok && active && lt.fast) {
#pragma unroll
        for (int u = 0; u < kBoxRows; u++) {
          float d = 0.f;
          if (u < n) {
            d = chunk_dot(lds128(st + u * lt.rowB + 16 * lane), L);
            if (lt.box_s) d *= lds32f(st + kBoxRows * kSliceWords * 4 + (u * lt.box_s + so) * 4);
          }
          acc[u] = d;
        }
      } else {
        float tmp[kBoxRows];  // local memory: the rarely used slow path keeps code small
#pragma unroll 1
        for (int u = 0; u < kBoxRows; u++)
          tmp[u] = (ok && active && u < n)
                       ? chunk_dot_slow(lds128(st + u * lt.rowB + 16 * lane), L, lt, P.h, COLI_DTYPE_F32,
                                        (size_t)k * P.I, d0 + u, c)
                       : 0.f;
#pragma unroll
        for (int u = 0; u < kBoxRows; u++) acc[u] = tmp[u];
      }
      __syncwarp();
      if (lane == 0) issue_next();
      if (!ok) {
        stop = true;
        set_error(P.err, COLI_E_TIMEOUT);
      }
      // lane l ends with the warp total of row l / 4 of the batch
      warp_transpose_reduce<kBoxRows>(acc, lane);
      if ((lane & 3) == 0 && (lane >> 2) < n) sm.part[warp][d0 - s0 + (lane >> 2)] = acc[0];
      b++;
    }
    if (rsk >= 0) sm.rscale[rsk][rsr] = rsv;
    const bool any_stop = named_sync_or(1, NC, stop);
    if (!any_stop && tid < nseg) {
      const int d = s0 + tid;
      float acc = 0.f;
      for (int kk = 0; kk < m; kk++) {
        if (!sm.ok[kk]) continue;
        float yk = 0.f;
        for (int wi = kk * wpe; wi < (kk + 1) * wpe; wi++) yk += sm.part[wi][tid];
        acc = fmaf(sm.wk[kk], yk * sm.rscale[kk][tid], acc);
      }
      if (P.resid) acc = res + acc;
      if (P.x_dtype == COLI_DTYPE_F32)
        static_cast<float*>(P.y)[d] = acc;
      else
        static_cast<uint16_t*>(P.y)[d] = f32_to_bf16_rn(acc);
    }
    named_sync(1, NC);
    if (any_stop) stop = true;
  }
  if (warp_on && lane == 0)  // never leave with TMA loads in flight into this warp's ring
    for (uint32_t q = issued > kWarpStages ? issued - kWarpStages : 0; q < issued; q++)
      if (q >= b) (void)mbar_wait(&bars[q % kWarpStages], (q / kWarpStages) & 1);
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
  const TensorDesc* Tdp = nullptr;
  int mode = SCALE_ROW, G = 1, gs = 0;
  uint32_t pitch = 0;
  const uint8_t* wbase = nullptr;
  const float* sbase = nullptr;
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
      if (route_ok) {
        Tdp = &P.table[e].t[T_DOWN];
        mode = Tdp->mode;
        G = Tdp->G;
        gs = Tdp->gs;
        pitch = Tdp->pitch;
        wbase = Tdp->w;
        sbase = Tdp->s;
      }
      load_chunk_f32(P.h, COLI_DTYPE_F32, (size_t)j * P.I, 32 * c, (has_chunk && route_ok) ? P.I : 0, hv);
      if (!make_limbs(hv, L)) set_error(P.err, COLI_E_NONFINITE);
    }
    float part[kDU];
    if (route_ok && has_chunk) {
      uint4 wv[kDU];
#pragma unroll
      for (int u = 0; u < kDU; u++)
        wv[u] = u < nb ? ldg_stream(wbase + (size_t)(d0 + u) * pitch + 16 * c)
                       : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
#pragma unroll
      for (int u = 0; u < kDU; u++) {
        float d;
        if (mode == SCALE_GENERIC) {
          d = u < nb ? chunk_dot_generic(wv[u], P.h, COLI_DTYPE_F32, (size_t)j * P.I, Tdp, d0 + u, c) : 0.f;
        } else {
          d = chunk_dot(wv[u], L);
          if (mode == SCALE_CHUNK && u < nb) d *= __ldg(sbase + (size_t)(d0 + u) * G + (32 * c) / gs);
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
      if (route_ok && mode == SCALE_ROW) yk *= __ldg(sbase + d0 + tid);
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
  if (D > COLI_MAX_GROUP_DIM) return fail(ctx, COLI_E_INVAL, "expert_group: D above COLI_MAX_GROUP_DIM");
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
  cudaError_t e;
  {
    const int W = (CD + 31) / 32;
    const int nt = W * 32;
    const size_t smem = gateup_smem_bytes(W, S);
    auto kern = nt <= 192 ? gateup_kernel<192> : gateup_kernel<256>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "gate/up smem attribute");
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nt, smem);
    // every CTA's range spans at most kRouteCache routes: (R I / grid) <= (kRouteCache - 2) I
    long long grid = (long long)ctx->num_sms * (occ > 0 ? occ : 1);
    const long long min_grid = ((long long)S * K + kRouteCache - 3) / (kRouteCache - 2);
    if (grid < min_grid) grid = min_grid;
    ProfScope prof(ctx, COLI_KERNEL_GATEUP);
    e = launch_k(kern, (int)grid, nt, smem, ctx->stream, true, P);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "gate/up launch");
  }
  const int TPE = (CI + 31) / 32 * 32;
  if (S == 1 && K * TPE <= 1024 && down_smem_bytes(K * TPE / 32) <= 220 * 1024) {
    const int nt = K * TPE;
    const size_t smem = down_smem_bytes(nt / 32);
    auto kern = nt <= 256 ? down_fused_kernel<256> : (nt <= 512 ? down_fused_kernel<512> : down_fused_kernel<1024>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "down smem attribute");
    int grid = ctx->num_sms;
    if (grid > D) grid = D;
    ProfScope prof(ctx, COLI_KERNEL_DOWN);
    e = launch_k(kern, grid, nt, smem, ctx->stream, true, P, TPE);
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
