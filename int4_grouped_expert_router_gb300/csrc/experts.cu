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
// power of two 2^q so that its largest magnitude lies in [2^21, 2^22), rounded to integers and
// split into three balanced signed bytes (x = l2 2^16 + l1 2^8 + l0). The nibble-by-limb
// products are then summed exactly in 32-bit integers with dp4a (four products per
// instruction), the offset 8 is removed through a precomputed -8 * sum(l), and the exact limb
// sums are combined in binary32 and scaled back by 2^-q. The chunk result therefore differs from
// the exact dot product of the given activations by two roundings of binary32 plus the
// activation quantisation: at most 2^-22 of the chunk's largest activation, per column.
// Chunk results are summed across the warp by a butterfly and across warps in a fixed order.
#include "coli_internal.h"
#include "dot.h"
#include "pipe.h"

namespace coli {

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
  int x_dtype;     // dtype of x and resid
  int y_dtype;     // dtype of y (x_dtype, or f32 for an issued partial sum)
  int S, D, I, K;
  const int32_t* idx;
  const float* w;
  const int32_t* n_sel;
  const ExpertDesc* table;
  const void* resid;
  void* y;
  float* h;        // [routes x I]
  int h_dtype;     // dtype of h (f32; the dense projection passes its activations here)
  float* yr;       // [routes x D] (S > 1)
  int* plan;       // pre[0..S] (written by CTA 0 of the gate/up kernel)
  int* err;
};

// ------------------------------------------------------------------------------------------
// Shared pieces of the two streaming kernels
//
// Every consumer warp owns one 512-byte column slice (32 chunks of 16 bytes) of the weight rows
// and streams it by itself: its lane 0 issues 2-D TMA loads of [kBoxRows rows x slice] boxes into
// the warp's own ring of shared-memory stages, a ring's depth of boxes ahead of the warp's
// compute. Warps never wait for each other while streaming; they meet only at the end of a
// segment of rows to add their slices' partial sums in a fixed order.
// ------------------------------------------------------------------------------------------

constexpr int kDStages = 4;  // stages per warp ring of the down kernel
#ifndef COLI_DOWN_PRE_STAGES
#define COLI_DOWN_PRE_STAGES 2
#endif
constexpr int kDPreStages = COLI_DOWN_PRE_STAGES;  // of them issued before the wait for h
constexpr int kSeg = 64;          // rows (down) or row pairs (gate/up) finished together
constexpr int kRouteCache = 16;   // routes resolved once into shared memory


// Everything a kernel needs about one tensor of a kept route, copied once into shared memory.
struct SlotTensor {
  const TensorDesc* d;  // in the device expert table (the TMA maps live there)
  const float* s;       // scales
  const uint8_t* w;     // packed rows
  uint32_t pitch;       // bytes per packed row
  int mode, G, gs, box_s, box_w, box_rows;
};

struct RouteSlot {
  SlotTensor ts[2];
  int t, ok;
};

__device__ __forceinline__ void fill_slot_tensor(SlotTensor& st, const TensorDesc* d) {
  prefetch_tensormap(&d->map_w);  // the first TMA load of this tensor follows shortly
  st.d = d;
  st.s = d->s;
  st.w = d->w;
  st.pitch = d->pitch;
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

// The slow paths (any even group size that is not a multiple of 32, or chunk scales that do not
// travel by TMA): the activation limbs stay in registers -- they are never passed by reference to
// an out-of-line function, which would move them to local memory for the whole kernel.
__device__ __forceinline__ float chunk_dot_slow(const uint4 wv, const Limbs& L, const LaneTensor& lt, const void* act,
                                                int dtype, size_t base, int row, int c) {
  if (lt.mode == SCALE_GENERIC) return chunk_dot_generic(wv, act, dtype, base, lt.d, row, c);
  return chunk_dot(wv, L) * __ldg(lt.s + (size_t)row * lt.G + lt.cg);
}


constexpr uint32_t kUpOff = kBoxRows * kSliceWords * 4;  // up box within a gate/up stage
constexpr uint32_t kScaleOff = 2 * kUpOff;               // gate scale box, then the up scale box

// Dot products of one batch from a stage of the warp's ring: acc[u] = gate row u, acc[kBoxRows + u]
// = up row u of this lane's chunk (scaled by chunk scales when those are staged; row scales are
// applied when the rows are finished). `st` is the stage base plus 16 * lane; n = rows of the batch
// inside the matrix (the fast paths compute all kBoxRows, the extra rows are never read back).
__device__ __forceinline__ void gateup_batch(float (&acc)[2 * kBoxRows], bool ok, bool has_chunk, bool row_scales,
                                             const LaneTensor& tg, const LaneTensor& tu, const uint8_t* st,
                                             const uint8_t* sgb, int warp, const Limbs& L, const GroupParams& P,
                                             int cur_tok, int i0, int n, int c) {
  if (ok && has_chunk && row_scales) {
#pragma unroll
    for (int u = 0; u < kBoxRows; u++) {
      acc[u] = chunk_dot(lds128(st + u * tg.rowB), L);
      acc[kBoxRows + u] = chunk_dot(lds128(st + kUpOff + u * tu.rowB), L);
    }
  } else if (ok && has_chunk && tg.fast && tu.fast) {
#pragma unroll
    for (int u = 0; u < kBoxRows; u++) {
      float dg = chunk_dot(lds128(st + u * tg.rowB), L);
      float du = chunk_dot(lds128(st + kUpOff + u * tu.rowB), L);
      if (tg.box_s) dg *= lds32f(sgb + (u * tg.box_s + tg.cg - tg.box_s * warp) * 4);
      if (tu.box_s) du *= lds32f(sgb + kBoxRows * kScaleBox * 4 + (u * tu.box_s + tu.cg - tu.box_s * warp) * 4);
      acc[u] = dg;
      acc[kBoxRows + u] = du;
    }
  } else {
    float tmp[2 * kBoxRows];  // local memory: the rarely used slow path keeps the code small
#pragma unroll 1
    for (int v = 0; v < 2 * kBoxRows; v++) {
      const int u = v % kBoxRows;
      const LaneTensor& lt = v < kBoxRows ? tg : tu;
      float d = 0.f;
      if (ok && has_chunk && u < n) {
        const uint4 wv = lds128(st + (v / kBoxRows) * kUpOff + u * lt.rowB);
        if (lt.fast)
          d = chunk_dot(wv, L) * (lt.box_s ? lds32f(sgb + (v / kBoxRows) * (kBoxRows * kScaleBox * 4) +
                                                    (u * lt.box_s + lt.cg - lt.box_s * warp) * 4)
                                           : 1.f);
        else
          d = chunk_dot_slow(wv, L, lt, P.x, P.x_dtype, (size_t)cur_tok * P.D, i0 + u, c);
      }
      tmp[v] = d;
    }
#pragma unroll
    for (int v = 0; v < 2 * kBoxRows; v++) acc[v] = tmp[v];
  }
}

// Issue the TMA loads of one batch (gate and up boxes, and staged chunk scales) into a stage.
__device__ __forceinline__ void gateup_issue(const RouteSlot& rs, uint8_t* st, uint64_t* bar, int warp, int i0) {
  const SlotTensor& g = rs.ts[0];
  const SlotTensor& u = rs.ts[1];
  uint32_t bytes = 2u * g.box_rows * g.box_w * 4;
  if (g.box_s) bytes += g.box_rows * g.box_s * 4;
  if (u.box_s) bytes += u.box_rows * u.box_s * 4;
  mbar_arrive_expect_tx(bar, bytes);
  const int x = kSliceWords * warp;
  tma_load_2d(st, &g.d->map_w, x, i0, bar);
  tma_load_2d(st + kUpOff, &u.d->map_w, x, i0, bar);
  if (g.box_s) tma_load_2d(st + kScaleOff, &g.d->map_s, g.box_s * warp, i0, bar);
  if (u.box_s) tma_load_2d(st + kScaleOff + kBoxRows * kScaleBox * 4, &u.d->map_s, u.box_s * warp, i0, bar);
}

// ------------------------------------------------------------------------------------------
// Gate + up dual GEMV with the SiLU(g) * u epilogue.
// Thread c of the CTA owns column chunk c (warp c / 32 owns slice c / 32) of every row and keeps
// that chunk of the activation in registers. A stage of a warp holds kBoxRows gate rows and
// kBoxRows up rows of its slice (and their chunk scales when those travel by TMA).
// Work items are batches of kBoxRows row pairs: route j owns batches covering its rows padded to
// a multiple of kBoxRows, so batch q is (route q / Bpr, first row kBoxRows (q % Bpr)) in closed
// form and a CTA owns a contiguous run of batches; segB batches (one row pair per thread of the
// CTA, at most kSeg) form a finishing segment.
//
// FUSED (S == 1, cooperative launch): the same kernel then runs the down projection. Every warp
// takes one (slot k, column slice) stream of a range of down rows; the ranges split D identically
// for every stream. Its first down boxes are staged into the warp's ring (the gate/up ring, free by
// then) before the grid-wide barrier that makes h complete, so the weight stream runs on while the
// last gate/up rows finish. After the barrier each warp turns its slice of h_k into limbs, streams
// its rows and writes per-row partial sums; the last of a range's streams to finish (a counter per
// range) adds them up in slot order -- the same order and arithmetic as the two-kernel path.
// ------------------------------------------------------------------------------------------

#ifndef COLI_GU_STAGES
#define COLI_GU_STAGES 3
#endif
#ifndef COLI_GU_MIN_CTAS
#define COLI_GU_MIN_CTAS 2
#endif
constexpr int kGUStages = COLI_GU_STAGES;    // stages per warp ring
constexpr int kGUMinCtas = COLI_GU_MIN_CTAS; // CTAs per SM the register budget is sized for

__device__ const float kOneF = 1.0f;         // stand-in scale for unconditional loads

__host__ __device__ constexpr uint32_t down_stage_bytes() { return kBoxRows * kSliceWords * 4 + kBoxRows * kScaleBox * 4; }

// stages of the fused kernel's down ring: it reuses the warp's gate/up ring
constexpr int kFDStages = (int)(kGUStages * (2u * kBoxRows * kSliceWords * 4 + 2u * kBoxRows * kScaleBox * 4) /
                                down_stage_bytes());

struct GateUpSmem {
  RouteSlot routes[kRouteCache];
  uint64_t bars[8][kGUStages];     // gate/up CTAs have at most 8 warps (D <= 8192)
  int e_spec[COLI_MAX_K];          // S == 1: the expert of each slot, read with n_sel
  // FUSED only
  uint64_t dbars[8][kFDStages];    // the warps' down rings
  SlotTensor dn[COLI_MAX_K];       // down tensor of each kept slot
  float wk[COLI_MAX_K];            // routing weight of each slot
  int dn_ok[COLI_MAX_K];
  int m;                           // kept slots
};

// Fused decode kernel: where the down phase keeps its cross-CTA state.
struct FusedParams {
  float* ypart;  // [K][nsl][D]: partial down rows of each (slot, column slice) stream
  int* sync;     // [0..1]: the grid barrier's 64-bit arrival count; [kSyncRanges + r]: arrivals at row range r
  int nsl;       // column slices of a down row: ceil(ceil(I / 32) / 32)
};
// followed in dynamic shared memory by the warps' rings, pg[W][kSeg], pu[W][kSeg], pre[S + 1]

static_assert((kBoxRows & (kBoxRows - 1)) == 0, "kBoxRows must be a power of two");

__host__ __device__ constexpr uint32_t gateup_stage_bytes() {
  // gate box + up box (kBoxRows x 512 B each) + two scale boxes (kBoxRows x kScaleBox floats)
  return 2u * kBoxRows * kSliceWords * 4 + 2u * kBoxRows * kScaleBox * 4;
}

// 2-D TMA writes need 128-byte-aligned shared-memory destinations: the rings start on a 128-byte
// boundary after the control block and every stage, box and scale box is a multiple of 128 bytes.
constexpr size_t kGUCtrlBytes = (sizeof(GateUpSmem) + 127) / 128 * 128;
static_assert(gateup_stage_bytes() % 128 == 0, "gate/up stage must keep 128-byte alignment");
static_assert((kBoxRows * kSliceWords * 4) % 128 == 0 && (kBoxRows * kScaleBox * 4) % 128 == 0,
              "TMA boxes must keep 128-byte alignment");

inline size_t gateup_smem_bytes(int W, int S) {
  return 128 + kGUCtrlBytes + (size_t)W * kGUStages * gateup_stage_bytes() + 2 * (size_t)W * kSeg * sizeof(float) +
         (size_t)(S + 1) * sizeof(int);
}

// Rows [d0, dend) of y, one row per lane at a time: residual + the sum over kept slots, in slot
// order, of w_k (row scale x the sum of the slot's NSL column-slice partials). Every load of a
// kRB-slot block is issued before its sums, from clamped (always valid) addresses, so the loads
// overlap instead of paying one L2 round trip each.
template <int NSL>
__device__ __forceinline__ void fused_finish_rows(const GroupParams& P, const FusedParams& F, const GateUpSmem& sm,
                                                  int m, int d0, int dend, int lane) {
  constexpr int kRB = 8;
  const int nsl = F.nsl;  // NSL >= nsl
  for (int d = d0 + lane; d < dend; d += 32) {
    float acc = 0.f;
    for (int k0 = 0; k0 < m; k0 += kRB) {
      float v[kRB][NSL], sv[kRB];
#pragma unroll
      for (int i = 0; i < kRB; i++) {
        const int kk = min(k0 + i, m - 1);
        const bool row_scale = sm.dn_ok[kk] && sm.dn[kk].mode == SCALE_ROW;
#pragma unroll
        for (int ss = 0; ss < NSL; ss++) v[i][ss] = __ldcg(F.ypart + ((size_t)kk * nsl + min(ss, nsl - 1)) * P.D + d);
        sv[i] = __ldg((row_scale ? sm.dn[kk].s : F.ypart) + d);
      }
#pragma unroll
      for (int i = 0; i < kRB; i++) {
        const int kk = k0 + i;
        if (kk < m && sm.dn_ok[kk]) {
          float yk = 0.f;
#pragma unroll
          for (int ss = 0; ss < NSL; ss++)
            if (ss < nsl) yk += v[i][ss];
          const float rs = sm.dn[kk].mode == SCALE_ROW ? sv[i] : 1.f;
          acc = fmaf(sm.wk[kk], yk * rs, acc);
        }
      }
    }
    float res = 0.f;
    if (P.resid) res = load_act(P.resid, P.x_dtype, d);
    if (P.resid) acc = res + acc;
    if (P.y_dtype == COLI_DTYPE_F32)
      static_cast<float*>(P.y)[d] = acc;
    else
      static_cast<uint16_t*>(P.y)[d] = f32_to_bf16_rn(acc);
  }
}

// Down phase of the fused decode kernel. `ring` is this warp's gate/up ring (drained by now).
__device__ __forceinline__ void fused_down_phase(const GroupParams& P, const FusedParams& F, GateUpSmem& sm,
                                                 uint8_t* ring, int W) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t DSB = down_stage_bytes();
  const int m = sm.m, nsl = F.nsl, T = m * nsl;  // streams: kept slots x column slices
  if (T == 0) {  // no kept route (uniform across the grid): y = residual
    for (int d = blockIdx.x * blockDim.x + tid; d < P.D; d += gridDim.x * blockDim.x) {
      float acc = 0.f;
      if (P.resid) acc = load_act(P.resid, P.x_dtype, d) + acc;
      if (P.y_dtype == COLI_DTYPE_F32)
        static_cast<float*>(P.y)[d] = acc;
      else
        static_cast<uint16_t*>(P.y)[d] = f32_to_bf16_rn(acc);
    }
    return;
  }
  // warp gw takes stream gw % T of row range gw / T; every stream splits D into the same NR ranges
  const int NW = gridDim.x * W, gw = blockIdx.x * W + warp;
  const int NR = min(NW / T, kMaxRanges);
  const int NBd = (P.D + kBoxRows - 1) / kBoxRows;  // row batches of a down matrix
  const int r = gw / T, pr = gw - r * T;
  const int k = pr / nsl, slice = pr - k * nsl;
  const bool task = r < NR;
  const int b0 = task ? (int)((long long)r * NBd / NR) : 0;
  const int b1 = task ? (int)((long long)(r + 1) * NBd / NR) : 0;
  const bool warp_on = task && sm.dn_ok[k];  // uniform per warp
  const SlotTensor& sl = sm.dn[warp_on ? k : 0];
  uint64_t* bars = sm.dbars[warp];
  const int CI = (P.I + 31) >> 5;
  const int c = slice * 32 + lane;
  const bool active = warp_on && c < CI;
  const uint32_t nbat = (uint32_t)(b1 - b0);
  uint32_t issued = 0;
  auto issue_next = [&]() {
    if (issued >= nbat) return;
    const uint32_t s = issued % kFDStages;
    uint8_t* st = ring + (size_t)s * DSB;
    const int d0 = (b0 + (int)issued) * kBoxRows;
    const uint32_t bytes = sl.box_rows * sl.box_w * 4 + (sl.box_s ? sl.box_rows * sl.box_s * 4 : 0);
    mbar_arrive_expect_tx(&bars[s], bytes);
    tma_load_2d(st, &sl.d->map_w, kSliceWords * slice, d0, &bars[s]);
    if (sl.box_s) tma_load_2d(st + kBoxRows * kSliceWords * 4, &sl.d->map_s, sl.box_s * slice, d0, &bars[s]);
    issued++;
  };
  __syncwarp();  // every lane is done with the gate/up ring
  if (warp_on && lane == 0)
    for (int s = 0; s < kFDStages; s++) issue_next();  // the down weights do not depend on h
  bool stop = !grid_barrier(reinterpret_cast<unsigned long long*>(F.sync));  // every row of h is written
  if (stop && tid == 0) set_error(P.err, COLI_E_TIMEOUT);

  LaneTensor lt;
  lane_tensor(lt, sl, c);
  const int so = lt.cg - lt.box_s * slice;  // lane's scale within the staged box
  float hv[32];
  Limbs L;
  load_chunk_f32(P.h, COLI_DTYPE_F32, (size_t)k * P.I, 32 * c, active ? P.I : 0, hv);
  if (!make_limbs(hv, L) && active) set_error(P.err, COLI_E_NONFINITE);
  float* yp = F.ypart + ((size_t)k * nsl + slice) * P.D;
  for (uint32_t b = 0; b < nbat; b++) {
    if (!warp_on || stop) break;
    const int d0 = (b0 + (int)b) * kBoxRows;
    const int n = min(kBoxRows, P.D - d0);
    const uint32_t s = b % kFDStages;
    const bool ok = mbar_wait(&bars[s], (b / kFDStages) & 1);
    const uint8_t* st = ring + (size_t)s * DSB;
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
    if (lane == 0 && ok) issue_next();
    if (!ok) {
      stop = true;
      set_error(P.err, COLI_E_TIMEOUT);
    }
    // lane l ends with the warp total of row l / (32 / kBoxRows) of the batch
    warp_transpose_reduce<kBoxRows>(acc, lane);
    constexpr int kSpread = 32 / kBoxRows;
    if ((lane & (kSpread - 1)) == 0 && (lane / kSpread) < n) yp[d0 + lane / kSpread] = acc[0];
  }
  if (warp_on && lane == 0)  // never leave with TMA loads in flight into the ring
    for (uint32_t q = issued > kFDStages ? issued - kFDStages : 0; q < issued; q++)
      (void)mbar_wait(&bars[q % kFDStages], (q / kFDStages) & 1);
  if (!task) return;

  // arrive at the range; the last of its T streams finishes its rows
  __threadfence();
  __syncwarp();
  int* ctr = F.sync + kSyncRanges + r;
  int last = 0;
  if (lane == 0) last = atomicAdd(ctr, 1) == T - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  if (lane == 0) atomicExch(ctr, 0);  // ready for the next launch
  __threadfence();
  const int d0 = b0 * kBoxRows, dend = min(b1 * kBoxRows, P.D);
  switch (nsl) {
    case 1: fused_finish_rows<1>(P, F, sm, m, d0, dend, lane); break;
    case 2: fused_finish_rows<2>(P, F, sm, m, d0, dend, lane); break;
    default: fused_finish_rows<kFusedMaxSlices>(P, F, sm, m, d0, dend, lane); break;
  }
}

template <bool FUSED>
__device__ __forceinline__ void gateup_body(const GroupParams& P, const FusedParams& F) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem_raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  const int C = (P.D + 31) >> 5;
  const int W = (C + 31) >> 5;
  const uint32_t SB = gateup_stage_bytes();
  GateUpSmem& sm = *reinterpret_cast<GateUpSmem*>(smem_raw);
  uint8_t* rings = smem_raw + kGUCtrlBytes;
  float* pg = reinterpret_cast<float*>(rings + (size_t)W * kGUStages * SB);
  float* pu = pg + (size_t)W * kSeg;
  int* pre = reinterpret_cast<int*>(pu + (size_t)W * kSeg);
  __shared__ int scratch32[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid;
  const bool has_chunk = c < C;
  uint8_t* ring = rings + (size_t)warp * kGUStages * SB;
  uint64_t* bars = sm.bars[warp];
  if (lane == 0) {
    for (int s = 0; s < kGUStages; s++) mbar_init(&bars[s], 1);
    if (FUSED)
      for (int s = 0; s < kFDStages; s++) mbar_init(&sm.dbars[warp][s], 1);
    mbar_fence_init();
  }
  // prologue overlapping the router's tail: activation limbs of token 0
  Limbs L;
  int cur_tok = 0;
  {
    float xv[32];
    load_chunk_f32(P.x, P.x_dtype, 0, 32 * c, has_chunk ? P.D : 0, xv);
    if (!make_limbs(xv, L) && has_chunk) set_error(P.err, COLI_E_NONFINITE);
  }
  griddep_wait();
  float w_slot = 0.f;
  if (P.S == 1 && tid < P.K) {  // same round trip as n_sel
    sm.e_spec[tid] = ld_cg_i32(P.idx + tid);
    if (FUSED) w_slot = ld_cg_f32(P.w + tid);
  }
  const int R = build_plan(P.n_sel, P.S, P.K, pre, scratch32);       // contains __syncthreads
  if (blockIdx.x == 0)
    for (int t = tid; t <= P.S; t += blockDim.x) P.plan[t] = pre[t];
  griddep_launch_dependents();

  const int Bpr = (P.I + kBoxRows - 1) / kBoxRows;  // batches per route
  const int segB = min(kSeg, W * 32) / kBoxRows;    // batches per finishing segment
  const long long NB = (long long)R * Bpr;
  const int qbeg = (int)((long long)blockIdx.x * NB / gridDim.x);
  const int qend = (int)((long long)(blockIdx.x + 1) * NB / gridDim.x);
  const int j_first = qbeg / Bpr;
  const int n_routes = qbeg < qend ? (qend - 1) / Bpr - j_first + 1 : 0;  // <= kRouteCache (launch sizing)
  if (n_routes > kRouteCache && tid == 0) set_error(P.err, COLI_E_INVAL);  // the launcher's grid rules this out
  const bool gu = qbeg < qend && n_routes <= kRouteCache;                   // uniform across the CTA
  if (FUSED && tid < P.K) {
    const int e = sm.e_spec[tid];
    const bool ok = tid < R && e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
    if (ok) fill_slot_tensor(sm.dn[tid], &P.table[e].t[T_DOWN]);
    sm.dn_ok[tid] = ok;
    sm.wk[tid] = ok ? w_slot : 0.f;
    if (tid == 0) sm.m = R;
  }
  if (gu && tid < n_routes) {
    const int j = j_first + tid;
    RouteSlot& rs = sm.routes[tid];
    if (P.S == 1) {
      const int e = sm.e_spec[j];
      rs.t = 0;
      rs.ok = e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
      if (rs.ok) {
        fill_slot_tensor(rs.ts[0], &P.table[e].t[T_GATE]);
        fill_slot_tensor(rs.ts[1], &P.table[e].t[T_UP]);
      }
    } else {
      resolve_slot(P, pre, j, T_GATE, T_UP, rs);
    }
    if (!rs.ok) set_error(P.err, COLI_E_ROUTE);
  }
  __syncthreads();
  if (gu) {
    // issue side of this warp's ring: kGUStages batches ahead of the compute (lane 0)
    int iq = qbeg, ij = j_first, ii = (qbeg - j_first * Bpr) * kBoxRows, istage = 0, issued = 0;
    auto issue_next = [&]() {
      while (iq < qend) {
        const int j = ij, i0 = ii;
        iq++;
        ii += kBoxRows;
        if (ii >= Bpr * kBoxRows) {
          ii = 0;
          ij++;
        }
        const RouteSlot& rs = sm.routes[j - j_first];
        if (!rs.ok) continue;
        gateup_issue(rs, ring + (size_t)istage * SB, &bars[istage], warp, i0);
        istage = istage + 1 == kGUStages ? 0 : istage + 1;
        issued++;
        return;
      }
    };
    if (lane == 0)
      for (int s = 0; s < kGUStages; s++) issue_next();

    // finaliser thread `tid` (< segB kBoxRows) of a segment: where its row pair goes and its row
    // scales, loaded when the segment starts and consumed when it ends
    float fg = 1.f, fu = 1.f;
    size_t hdst = 0;
    bool fin_ok = false;
    auto prefetch_finaliser = [&](int q0) {
      const int qq = q0 + tid / kBoxRows;
      const int jj = qq / Bpr, i = (qq - jj * Bpr) * kBoxRows + tid % kBoxRows;
      fin_ok = tid < segB * kBoxRows && qq < qend && i < P.I && sm.routes[jj - j_first].ok;
      const RouteSlot& r = sm.routes[fin_ok ? jj - j_first : 0];
      hdst = (size_t)jj * P.I + i;
      fg = __ldg((fin_ok && r.ts[0].mode == SCALE_ROW) ? r.ts[0].s + i : &kOneF);
      fu = __ldg((fin_ok && r.ts[1].mode == SCALE_ROW) ? r.ts[1].s + i : &kOneF);
    };

    // ---------------- compute ----------------
    int cur_slot = -1;
    LaneTensor tg, tu;
    bool stop = false, row_scales = false;
    int stage = 0;
    uint32_t phase = 0;
    int j = j_first, i0 = (qbeg - j_first * Bpr) * kBoxRows;
    for (int qs = qbeg; qs < qend; qs += segB) {
      const int qe = min(qs + segB, qend);
      prefetch_finaliser(qs);
      for (int q = qs; q < qe; q++) {
        const int slot = j - j_first;
        if (sm.routes[slot].ok) {
          if (slot != cur_slot) {
            cur_slot = slot;
            const RouteSlot& rs = sm.routes[slot];
            lane_tensor(tg, rs.ts[0], c);
            lane_tensor(tu, rs.ts[1], c);
            row_scales = tg.fast && tu.fast && !tg.box_s && !tu.box_s;
            if (rs.t != cur_tok) {
              cur_tok = rs.t;
              float xv[32];
              load_chunk_f32(P.x, P.x_dtype, (size_t)cur_tok * P.D, 32 * c, has_chunk ? P.D : 0, xv);
              if (!make_limbs(xv, L) && has_chunk) set_error(P.err, COLI_E_NONFINITE);
            }
          }
          const bool ok = !stop && mbar_wait(&bars[stage], phase);
          const uint8_t* st = ring + (size_t)stage * SB + 16 * lane;
          float acc[2 * kBoxRows];  // gate rows 0..3, then up rows 0..3
          gateup_batch(acc, ok, has_chunk, row_scales, tg, tu, st, ring + (size_t)stage * SB + kScaleOff, warp, L, P,
                       cur_tok, i0, min(kBoxRows, P.I - i0), c);
          __syncwarp();
          if (lane == 0 && ok) issue_next();  // refill the stage just consumed
          if (!ok && !stop) {
            stop = true;
            set_error(P.err, COLI_E_TIMEOUT);
          }
          if (++stage == kGUStages) {
            stage = 0;
            phase ^= 1u;
          }
          // lane l ends with the warp total of value l / 4: gate row v (v < 4) or up row v - 4.
          // Box rows at and beyond I (zero-filled by TMA) give values that are never read back.
          warp_transpose_reduce<2 * kBoxRows>(acc, lane);
          if ((lane & 3) == 0) {
            const int v = lane >> 2;
            (v < kBoxRows ? pg : pu)[warp * kSeg + (q - qs) * kBoxRows + (v & (kBoxRows - 1))] = acc[0];
          }
        }
        i0 += kBoxRows;
        if (i0 >= Bpr * kBoxRows) {
          i0 = 0;
          j++;
        }
      }
      // segment end: finish its rows
      const bool any_stop = named_sync_or(1, W * 32, stop);
      if (!any_stop && fin_ok) {
        float g = 0.f, u = 0.f;
        for (int wi = 0; wi < W; wi++) {
          g += pg[wi * kSeg + tid];
          u += pu[wi * kSeg + tid];
        }
        P.h[hdst] = silu_mul(g * fg, u * fu);
      }
      named_sync(1, W * 32);  // the partial buffers are reused by the next segment
      if (any_stop) stop = true;
    }
    // never leave with TMA loads in flight into this warp's ring (the last issued phases)
    if (lane == 0)
      for (int q = issued > kGUStages ? issued - kGUStages : 0; q < issued; q++)
        (void)mbar_wait(&bars[q % kGUStages], (q / kGUStages) & 1);
  }  // gu
  if constexpr (FUSED) fused_down_phase(P, F, sm, rings + (size_t)warp * kGUStages * SB, W);
}

template <int MAXT>
__global__ void __launch_bounds__(MAXT, MAXT <= 192 ? kGUMinCtas : 1) gateup_kernel(GroupParams P) {
  gateup_body<false>(P, FusedParams{});
}

// S == 1: the whole expert FFN (gate/up, down, weighting and the reduce) in one cooperative launch.
template <int MAXT>
__global__ void __launch_bounds__(MAXT, MAXT <= 192 ? kGUMinCtas : 1) decode_ffn_kernel(GroupParams P, FusedParams F) {
  gateup_body<true>(P, F);
}

// ------------------------------------------------------------------------------------------
// S == 1: down GEMV of every kept slot, weighting and the slot-ordered reduce in one kernel.
// Threads (k, c): slot k = tid / TPE owns column chunk c = tid % TPE of its expert's down rows,
// with that chunk of h_k in registers; each warp streams its own slice of its expert's rows. The
// weight stream does not depend on the gate/up kernel, so it starts before that kernel ends.
// ------------------------------------------------------------------------------------------

struct DownSmem {
  uint64_t bars[32][kDStages];
  float part[32][kSeg];
  float rscale[COLI_MAX_K][kSeg];
  float wk[COLI_MAX_K];
  SlotTensor st[COLI_MAX_K];
  int ok[COLI_MAX_K];
};

constexpr size_t kDCtrlBytes = (sizeof(DownSmem) + 127) / 128 * 128;
static_assert(down_stage_bytes() % 128 == 0, "down stage must keep 128-byte alignment");

inline size_t down_smem_bytes(int nwarps) {
  return 128 + kDCtrlBytes + (size_t)nwarps * kDStages * down_stage_bytes();
}

template <int MAXT>
__global__ void __launch_bounds__(MAXT, 1) down_reduce_kernel(GroupParams P, int TPE) {
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
  uint8_t* ring = smem_raw + kDCtrlBytes + (size_t)warp * kDStages * SB;
  uint64_t* bars = sm.bars[warp];

  // routes of token 0 (written by the router, complete before the gate/up kernel started); the
  // count, ids and weights are read in one round trip
  int m = P.n_sel ? ld_cg_i32(P.n_sel) : P.K;
  const int e_slot = tid < P.K ? ld_cg_i32(P.idx + tid) : -1;
  const float w_slot = tid < P.K ? ld_cg_f32(P.w + tid) : 0.f;
  m = m < 0 ? 0 : (m > P.K ? P.K : m);
  if (lane == 0) {
    for (int s = 0; s < kDStages; s++) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  if (tid < P.K) {
    bool ok = false;
    if (tid < m) {
      ok = e_slot >= 0 && e_slot < COLI_MAX_EXPERTS && P.table[e_slot].valid;
      if (ok) fill_slot_tensor(sm.st[tid], &P.table[e_slot].t[T_DOWN]);
      else set_error(P.err, COLI_E_ROUTE);
    }
    sm.ok[tid] = ok;
    sm.wk[tid] = ok ? w_slot : 0.f;
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
    const uint32_t s = issued % kDStages;
    uint8_t* st = ring + (size_t)s * SB;
    const int d0 = d_begin + (int)issued * kBoxRows;
    uint32_t bytes = sl->box_rows * sl->box_w * 4 + (sl->box_s ? sl->box_rows * sl->box_s * 4 : 0);
    mbar_arrive_expect_tx(&bars[s], bytes);
    tma_load_2d(st, &sl->d->map_w, kSliceWords * slice, d0, &bars[s]);
    if (sl->box_s) tma_load_2d(st + kBoxRows * kSliceWords * 4, &sl->d->map_s, sl->box_s * slice, d0, &bars[s]);
    issued++;
  };
  if (warp_on && lane == 0)
    for (int s = 0; s < kDPreStages; s++) issue_next();  // the weight stream starts before h is ready

  LaneTensor lt;
  lane_tensor(lt, *sl, c);
  const int so = lt.cg - lt.box_s * slice;  // lane's scale within the staged box
  griddep_wait();  // h is written by the gate/up kernel
  float hv[32];
  Limbs L;
  load_chunk_f32(P.h, P.h_dtype, (size_t)k * P.I, 32 * c, active ? P.I : 0, hv);
  if (!make_limbs(hv, L) && active) set_error(P.err, COLI_E_NONFINITE);
  if (warp_on && lane == 0)  // the rest of the ring once h has arrived (its loads go first)
    for (int s = kDPreStages; s < kDStages; s++) issue_next();

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
      const uint32_t s = b % kDStages;
      const bool ok = mbar_wait(&bars[s], (b / kDStages) & 1);
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
                       ? chunk_dot_slow(lds128(st + u * lt.rowB + 16 * lane), L, lt, P.h, P.h_dtype,
                                        (size_t)k * P.I, d0 + u, c)
                       : 0.f;
#pragma unroll
        for (int u = 0; u < kBoxRows; u++) acc[u] = tmp[u];
      }
      __syncwarp();
      if (lane == 0 && ok) issue_next();
      if (!ok) {
        stop = true;
        set_error(P.err, COLI_E_TIMEOUT);
      }
      // lane l ends with the warp total of row l / (32 / kBoxRows) of the batch
      warp_transpose_reduce<kBoxRows>(acc, lane);
      constexpr int kSpread = 32 / kBoxRows;
      if ((lane & (kSpread - 1)) == 0 && (lane / kSpread) < n) sm.part[warp][d0 - s0 + lane / kSpread] = acc[0];
      b++;
    }
    if (rsk >= 0) sm.rscale[rsk][rsr] = rsv;
    // blocks with fewer threads than K nseg scale cells or nseg rows (K ceil(I/1024) 32 < 64) take the rest in strides
    for (int i = tid + NC; i < P.K * nseg; i += NC) {
      const int kk = i / nseg, r = i - kk * nseg;
      sm.rscale[kk][r] = (kk < m && sm.ok[kk] && sm.st[kk].mode == SCALE_ROW) ? __ldg(sm.st[kk].s + s0 + r) : 1.f;
    }
    const bool any_stop = named_sync_or(1, NC, stop);
    for (int r = tid; !any_stop && r < nseg; r += NC) {
      const int d = s0 + r;
      float acc = 0.f;
      for (int kk = 0; kk < m; kk++) {
        if (!sm.ok[kk]) continue;
        float yk = 0.f;
        for (int wi = kk * wpe; wi < (kk + 1) * wpe; wi++) yk += sm.part[wi][r];
        acc = fmaf(sm.wk[kk], yk * sm.rscale[kk][r], acc);
      }
      if (P.resid) acc = (r == tid ? res : load_act(P.resid, P.x_dtype, d)) + acc;
      if (P.y_dtype == COLI_DTYPE_F32)
        static_cast<float*>(P.y)[d] = acc;
      else
        static_cast<uint16_t*>(P.y)[d] = f32_to_bf16_rn(acc);
    }
    named_sync(1, NC);
    if (any_stop) stop = true;
  }
  if (warp_on && lane == 0)  // never leave with TMA loads in flight into this warp's ring
    for (uint32_t q = issued > kDStages ? issued - kDStages : 0; q < issued; q++)
      (void)mbar_wait(&bars[q % kDStages], (q / kDStages) & 1);
}

// ------------------------------------------------------------------------------------------
// S > 1: down GEMV per kept route into yr, then a slot-ordered combine per token.
// ------------------------------------------------------------------------------------------

constexpr int kDU = 4;  // rows per batch of the route-parallel down kernel

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
    if (P.y_dtype == COLI_DTYPE_F32)
      static_cast<float*>(P.y)[i] = acc;
    else
      static_cast<uint16_t*>(P.y)[i] = f32_to_bf16_rn(acc);
  }
}

// ------------------------------------------------------------------------------------------
// Dense int4 projection: y[t, o] = resid[t, o] + sum_i W[o, i] x[t, i] for S tokens.
//
// The same block-fixed-point dot product as the expert kernels. A thread owns one 16-byte chunk
// (32 columns) of every row; a CTA takes a contiguous range of (token, kLinRows-row batch) items,
// ordered token-major so a token's limbs are computed once per CTA. Each batch's rows are loaded
// from HBM with streaming loads, the next batch's issued before the current batch's products, so a
// CTA of two batches has all its rows in flight in one round trip. The products are reduced
// across the warp and the warp totals parked in shared memory; every kLinSeg batches the CTA adds
// the warps' totals in warp order and writes the finished rows.
// ------------------------------------------------------------------------------------------

struct LinearParams {
  const void* x;      // [S x I], x_dtype
  const void* resid;  // [S x O], x_dtype, or NULL
  void* y;            // [S x O], x_dtype
  int x_dtype;
  int S, O, I;
  int* err;
};

constexpr int kLinRows = 8;  // rows per batch
constexpr int kLinSeg = 8;   // batches finished together

// Position of a (token, row batch) item, advanced one item at a time (no divisions in the loops).
struct LinPos {
  int t, ob;  // token, row batch within the token
  __device__ __forceinline__ void next(int Bo) {
    if (++ob == Bo) {
      ob = 0;
      ++t;
    }
  }
};

template <int MAXT>
__global__ void __launch_bounds__(MAXT) linear_kernel(LinearParams P, const __grid_constant__ TensorDesc T) {
  __shared__ float red[MAXT / 32][kLinSeg * kLinRows];
  __shared__ int row_of[kLinSeg][2];  // (token, first row) of each batch of the segment
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int CI = (P.I + 31) >> 5;
  const int c = tid;
  const bool has_chunk = c < CI;
  const int Bo = (P.O + kLinRows - 1) / kLinRows;  // row batches per token
  const long long NB = (long long)P.S * Bo;        // < 2^31 (S <= 65536, O <= 32768)
  const int q0 = (int)((long long)blockIdx.x * NB / gridDim.x);
  const int q1 = (int)((long long)(blockIdx.x + 1) * NB / gridDim.x);
  const uint4 zero_w = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);  // nibbles 8: value 0
  auto load_batch = [&](bool live, const LinPos& ps, uint4 (&wv)[kLinRows]) {
    const int o0 = ps.ob * kLinRows;
#pragma unroll
    for (int u = 0; u < kLinRows; u++)
      wv[u] = (has_chunk && live && o0 + u < P.O) ? ldg_stream(T.w + (size_t)(o0 + u) * T.pitch + 16 * c) : zero_w;
  };
  LinPos pos{q0 / Bo, q0 % Bo};  // the batch being computed
  LinPos ahead = pos;            // the batch whose rows are loaded next
  Limbs L;
  int cur_t = -1;
  uint4 wnext[kLinRows];
  load_batch(q0 < q1, ahead, wnext);
  ahead.next(Bo);
  for (int qs = q0; qs < q1; qs += kLinSeg) {
    const int nq = min(kLinSeg, q1 - qs);
    for (int b = 0; b < nq; b++) {
      const int t = pos.t, o0 = pos.ob * kLinRows;
      if (tid == 0) {
        row_of[b][0] = t;
        row_of[b][1] = o0;
      }
      uint4 wv[kLinRows];
#pragma unroll
      for (int u = 0; u < kLinRows; u++) wv[u] = wnext[u];
      load_batch(qs + b + 1 < q1, ahead, wnext);
      ahead.next(Bo);
      if (t != cur_t) {  // uniform across the CTA
        cur_t = t;
        float xv[32];
        load_chunk_f32(P.x, P.x_dtype, (size_t)t * P.I, 32 * c, has_chunk ? P.I : 0, xv);
        if (!make_limbs(xv, L) && has_chunk) set_error(P.err, COLI_E_NONFINITE);
      }
      float part[kLinRows];
#pragma unroll
      for (int u = 0; u < kLinRows; u++) {
        float d = 0.f;
        if (has_chunk && o0 + u < P.O) {
          if (T.mode == SCALE_GENERIC) {
            d = chunk_dot_generic(wv[u], P.x, P.x_dtype, (size_t)t * P.I, &T, o0 + u, c);
          } else {
            d = chunk_dot(wv[u], L);
            if (T.mode == SCALE_CHUNK) d *= __ldg(T.s + (size_t)(o0 + u) * T.G + (32 * c) / T.gs);
          }
        }
        part[u] = d;
      }
      // lane l ends with the warp total of row l / (32 / kLinRows) of the batch
      warp_transpose_reduce<kLinRows>(part, lane);
      if ((lane & (32 / kLinRows - 1)) == 0) red[warp][b * kLinRows + lane / (32 / kLinRows)] = part[0];
      pos.next(Bo);
    }
    __syncthreads();
    for (int r = tid; r < nq * kLinRows; r += blockDim.x) {
      const int t = row_of[r / kLinRows][0];
      const int o = row_of[r / kLinRows][1] + r % kLinRows;
      if (o >= P.O) continue;
      float acc = 0.f;
      for (int wi = 0; wi < nwarps; wi++) acc += red[wi][r];
      if (T.mode == SCALE_ROW) acc *= __ldg(T.s + o);
      const size_t i = (size_t)t * P.O + o;
      if (P.resid) acc = load_act(P.resid, P.x_dtype, i) + acc;
      if (P.x_dtype == COLI_DTYPE_F32)
        static_cast<float*>(P.y)[i] = acc;
      else
        static_cast<uint16_t*>(P.y)[i] = f32_to_bf16_rn(acc);
    }
    __syncthreads();  // red and row_of are reused by the next segment
  }
}

// ------------------------------------------------------------------------------------------
// Resident take: the issued groups' partial sums, in issue order, joined to the residual.
// ------------------------------------------------------------------------------------------

__global__ void take_kernel(const float* __restrict__ slots, int n, long long cells, const void* resid, int dtype,
                            void* y) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < cells; i += (long long)gridDim.x * blockDim.x) {
    float acc = __ldcg(slots + i);
    for (int j = 1; j < n; j++) acc = __fadd_rn(acc, __ldcg(slots + (size_t)j * cells + i));
    if (resid) acc = load_act(resid, dtype, i) + acc;
    if (dtype == COLI_DTYPE_F32)
      static_cast<float*>(y)[i] = acc;
    else
      static_cast<uint16_t*>(y)[i] = f32_to_bf16_rn(acc);
  }
}

int launch_take(coli_ctx* ctx, int S, int D, int n, const void* resid, int dtype, void* y) {
  const long long cells = (long long)S * D;
  int grid = (int)((cells + 255) / 256);
  if (grid > 4 * ctx->num_sms) grid = 4 * ctx->num_sms;
  {
    ProfScope prof(ctx, COLI_KERNEL_COMBINE);
    take_kernel<<<grid, 256, 0, ctx->stream>>>(ctx->slots, n, cells, resid, dtype, y);
  }
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? COLI_OK : cuda_fail(ctx, e, "take launch");
}

// ------------------------------------------------------------------------------------------
// Host launcher
// ------------------------------------------------------------------------------------------


__global__ void coop_probe_kernel(int* p) {
  if (p) *p = 0;
}

int probe_coop_mode(coli_ctx* ctx) {
  int coop = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, ctx->device) != cudaSuccess || !coop) {
    (void)cudaGetLastError();
    return 0;
  }
  cudaStream_t st;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  int mode = 0;
  for (int m = 2; m >= 1 && mode == 0; m--) {
    cudaError_t e = launch_k(coop_probe_kernel, 1, 32, 0, st, m == 2, true, (int*)nullptr);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) mode = m;
    (void)cudaGetLastError();
  }
  cudaStreamDestroy(st);
  return mode;
}

int launch_expert_group(coli_ctx* ctx, const void* x, int x_dtype, int S, const int32_t* idx, const float* w,
                        const int32_t* n_sel, int K, const void* resid, void* y, int y_dtype) {
  if (prefill_eligible(ctx, x, S, K, x_dtype)) return launch_prefill(ctx, x, S, idx, w, n_sel, K, resid, y, y_dtype);
  if (stream_eligible(ctx, S)) return launch_stream_ffn(ctx, x, x_dtype, idx, w, n_sel, K, resid, y, y_dtype);
  if (S > COLI_MAX_GROUP_TOKENS) return fail(ctx, COLI_E_INVAL, "expert_group: S above COLI_MAX_GROUP_TOKENS");
  const int D = ctx->table_D, I = ctx->table_I;
  if (D > COLI_MAX_GROUP_DIM) return fail(ctx, COLI_E_INVAL, "expert_group: D above COLI_MAX_GROUP_DIM");
  const int CD = (D + 31) / 32, CI = (I + 31) / 32;
  const int W = (CD + 31) / 32;  // gate/up warps per CTA
  const int nt_gu = W * 32;
  const size_t gu_smem = gateup_smem_bytes(W, S);
  cudaError_t e;
  // S == 1: gate/up and down in one cooperative kernel, when its whole grid fits on the device
  const int nsl = (CI + 31) / 32;
  bool fused = false;
  int fused_grid = 0;
  if (S == 1 && ctx->decode_fused && ctx->coop_mode > 0 && nsl <= kFusedMaxSlices) {
    auto kern = nt_gu <= 192 ? decode_ffn_kernel<192> : decode_ffn_kernel<256>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu_smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "fused decode smem attribute");
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nt_gu, gu_smem) != cudaSuccess) {
      (void)cudaGetLastError();
      occ = 0;
    }
    fused_grid = ctx->num_sms * occ;
    fused = occ > 0 && (long long)fused_grid * W >= (long long)K * nsl;
  }
  // otherwise the down projection: S == 1 with all slots' threads in one CTA (down_reduce_kernel),
  // else per-route rows into yr and a combine
  const int TPE = (CI + 31) / 32 * 32;
  const bool down_reduce = S == 1 && K * TPE <= 1024 && down_smem_bytes(K * TPE / 32) <= 220 * 1024;
  const size_t R = (size_t)S * K;
  const size_t h_bytes = align_up(R * I * sizeof(float), 256);
  const size_t yr_bytes = (!fused && !down_reduce) ? align_up(R * D * sizeof(float), 256) : 0;
  const size_t yp_bytes = fused ? align_up((size_t)K * nsl * D * sizeof(float), 256) : 0;
  const size_t plan_bytes = align_up((size_t)(S + 1) * sizeof(int), 256);
  int rc = ensure_workspace(ctx, h_bytes + yr_bytes + yp_bytes + plan_bytes);
  if (rc != COLI_OK) return rc;
  GroupParams P;
  P.x = x;
  P.x_dtype = x_dtype;
  P.y_dtype = y_dtype;
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
  P.h_dtype = COLI_DTYPE_F32;
  P.yr = reinterpret_cast<float*>(ctx->ws.base + h_bytes);
  P.plan = reinterpret_cast<int*>(ctx->ws.base + h_bytes + yr_bytes + yp_bytes);
  P.err = ctx->d_status;

  if (fused) {
    FusedParams F;
    F.ypart = reinterpret_cast<float*>(ctx->ws.base + h_bytes + yr_bytes);
    F.sync = ctx->d_status + kSyncBase;
    F.nsl = nsl;
    auto kern = nt_gu <= 192 ? decode_ffn_kernel<192> : decode_ffn_kernel<256>;
    ProfScope prof(ctx, COLI_KERNEL_GATEUP);
    e = launch_k(kern, fused_grid, nt_gu, gu_smem, ctx->stream, ctx->coop_mode == 2, true, P, F);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "fused decode launch");
    return COLI_OK;
  }
  {
    auto kern = nt_gu <= 192 ? gateup_kernel<192> : gateup_kernel<256>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu_smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "gate/up smem attribute");
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nt_gu, gu_smem);
    // every CTA's range spans at most kRouteCache routes: (R I / grid) <= (kRouteCache - 2) I
    long long grid = (long long)ctx->num_sms * (occ > 0 ? occ : 1);
    const long long min_grid = ((long long)S * K + kRouteCache - 3) / (kRouteCache - 2);
    if (grid < min_grid) grid = min_grid;
    ProfScope prof(ctx, COLI_KERNEL_GATEUP);
    e = launch_k(kern, (int)grid, nt_gu, gu_smem, ctx->stream, true, false, P);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "gate/up launch");
  }
  if (down_reduce) {
    const int nt = K * TPE;
    const size_t smem = down_smem_bytes(nt / 32);
    // block sizes between 512 and 1024 (K = 9..12 slots of 64 threads) get their own register budgets
    auto kern = nt <= 256   ? down_reduce_kernel<256>
                : nt <= 512 ? down_reduce_kernel<512>
                : nt <= 640 ? down_reduce_kernel<640>
                : nt <= 768 ? down_reduce_kernel<768>
                            : down_reduce_kernel<1024>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "down smem attribute");
    int grid = ctx->num_sms;
    if (grid > D) grid = D;
    ProfScope prof(ctx, COLI_KERNEL_DOWN);
    e = launch_k(kern, grid, nt, smem, ctx->stream, true, false, P, TPE);
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

int launch_linear(coli_ctx* ctx, const TensorDesc& T, const ExpertDesc* solo, const void* x, int x_dtype, int S,
                  const void* resid, void* y) {
  const int CI = (T.cols + 31) / 32;
  const int TPE = (CI + 31) / 32 * 32;
  if (S == 1 && solo && down_smem_bytes(TPE / 32) <= 220 * 1024) {
    // one token: the down kernel's per-warp TMA rings over a one-slot route {expert 0 of `solo`, weight 1},
    // with the activations in place of h
    GroupParams G{};
    G.x = x;
    G.x_dtype = x_dtype;
    G.y_dtype = x_dtype;
    G.S = 1;
    G.D = T.rows;
    G.I = T.cols;
    G.K = 1;
    G.idx = ctx->d_solo_route;
    G.w = reinterpret_cast<const float*>(ctx->d_solo_route + 1);
    G.n_sel = nullptr;
    G.table = solo;
    G.resid = resid;
    G.y = y;
    G.h = const_cast<float*>(static_cast<const float*>(x));
    G.h_dtype = x_dtype;
    G.err = ctx->d_status;
    const size_t smem = down_smem_bytes(TPE / 32);
    auto kern = TPE <= 256 ? down_reduce_kernel<256> : (TPE <= 512 ? down_reduce_kernel<512> : down_reduce_kernel<1024>);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return cuda_fail(ctx, e, "linear smem attribute");
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, TPE, smem) != cudaSuccess) {
      (void)cudaGetLastError();
      occ = 1;
    }
    int grid = ctx->num_sms * (occ > 0 ? occ : 1);
    if (grid > T.rows) grid = T.rows;
    ProfScope prof(ctx, COLI_KERNEL_LINEAR);
    e = launch_k(kern, grid, TPE, smem, ctx->stream, false, false, G, TPE);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "linear launch");
    return COLI_OK;
  }
  LinearParams P;
  P.x = x;
  P.resid = resid;
  P.y = y;
  P.x_dtype = x_dtype;
  P.S = S;
  P.O = T.rows;
  P.I = T.cols;
  P.err = ctx->d_status;
  const int nt = TPE;
  auto kern = nt <= 256 ? linear_kernel<256> : (nt <= 512 ? linear_kernel<512> : linear_kernel<1024>);
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nt, 0) != cudaSuccess) {
    (void)cudaGetLastError();
    occ = 1;
  }
  // at least two row batches per CTA: a CTA computes its token's limbs once per range
  const long long NB = (long long)S * ((T.rows + kLinRows - 1) / kLinRows);
  long long grid = (long long)ctx->num_sms * (occ > 0 ? occ : 1);
  if (grid > (NB + 1) / 2) grid = (NB + 1) / 2;
  if (grid < 1) grid = 1;
  ProfScope prof(ctx, COLI_KERNEL_LINEAR);
  kern<<<(int)grid, nt, 0, ctx->stream>>>(P, T);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "linear launch");
  return COLI_OK;
}

}  // namespace coli
