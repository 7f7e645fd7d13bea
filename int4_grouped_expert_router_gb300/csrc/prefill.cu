// Grouped int4 expert FFN on the tensor cores, for batches with many routed rows per expert
// (prefill). The routed rows are grouped by expert; per expert, the gate and up projections are
// bf16 GEMMs against the expert's block of activation rows, SiLU(gate) * up is written in bf16,
// the down projection is a second GEMM, and a slot-ordered combine adds the weighted expert
// outputs to the residual.
//
// Sources: c/backend_cuda.cu commit history -- commit "The TC_W4A16 branch ..." (a tensor-core
// W4A16 path gated on rows per expert, int4 weights dequantised to 16-bit for the contraction),
// commit "grouped MoE kernels were per-row-only" (per-row and per-group scales, mixed members);
// PR #434 "COLI_CUDA_RESID=1", section "What" (per-expert weighting, fixed-order reduce).
//
// Arithmetic. Weights enter the tensor core as bf16(bf16(s) (n - 8)) (s the row's or the group's
// scale, n the stored nibble); activations and SiLU(g) * u as bf16; products are accumulated in
// f32 in tensor memory; the combine sums the slots in slot order in f32.
//
// GEMM orientation. The weight rows are the MMA's M side (tiles of 128 rows) and an expert's
// tokens are its N side (16..128 columns), so the accumulator is D^T = W X^T in tensor memory.
// Both operands are K-major bf16 tiles of 64 columns in the 128-byte-swizzled layout: the
// activations are staged by TMA; the weights are staged packed by TMA and dequantised into that
// layout by converter warps. Within every 8-column group the dequantiser emits the columns in the
// order 0 4 1 5 2 6 3 7; the activation rows (and h, the down GEMM's activations) are stored in the
// same order, which leaves every dot product unchanged.
#include <cuda_bf16.h>

#include "coli_internal.h"
#include "pipe.h"
#include "tc.h"

namespace coli {

constexpr int kPfRows = 128;    // tokens (GEMM N) per work entry
constexpr int kPfPad = 16;      // per-entry token blocks are padded to a multiple of 16
constexpr int kPfKTile = 64;    // K columns per pipeline stage
constexpr int kPfStages = 3;
constexpr int kPfConvWarps = 8;  // warps 2..9 convert; warps 4..7 also drain the accumulators
constexpr int kPfThreads = (2 + kPfConvWarps) * 32;
constexpr uint32_t kPfTileBytes = kTcRows * 128;       // one bf16 operand tile: 128 rows x 128 bytes
constexpr uint32_t kPfPackedBytes = kTcRows * kTcWords * 4;  // one packed int4 weight tile

// position of column c (0..7) of an 8-column group in the tensor-core K order
__host__ __device__ constexpr int pf_perm8(int c) { return c < 4 ? 2 * c : 2 * (c - 4) + 1; }

struct PfEntry {
  int e;     // expert
  int row0;  // first row in the expert-grouped activation matrix
  int n;     // tokens (<= kPfRows)
  int npad;  // n rounded up to kPfPad (the MMA N)
};

// ------------------------------------------------------------------------------------------
// Route grouping: per expert, the kept routes (t, k) in increasing t k order.
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ bool pf_route_is(const int32_t* idx, const int32_t* n_sel, int K, int r, int SK, int e) {
  if (r >= SK) return false;
  const int t = r / K, k = r - t * K;
  int ns = n_sel ? __ldg(n_sel + t) : K;
  ns = ns < 0 ? 0 : (ns > K ? K : ns);
  return k < ns && __ldg(idx + r) == e;
}

// One warp per expert: kept routes naming it (0 for an expert without a valid table entry).
__global__ void pf_count_kernel(const int32_t* idx, const int32_t* n_sel, int S, int K, int E, const ExpertDesc* table,
                                int* cnt) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (e >= E) return;
  const int SK = S * K;
  int c = 0;
  if (table[e].valid)
    for (int base = 0; base < SK; base += 32) c += __popc(__ballot_sync(0xffffffffu, pf_route_is(idx, n_sel, K, base + lane, SK, e)));
  if (lane == 0) cnt[e] = c;
}

// One CTA: row offsets of every expert's padded blocks, the work entries, the total rows, and
// pos[] = src[] = -1.
__global__ void pf_plan_kernel(const int* cnt, int E, int SK, int R_max, int* row_off, PfEntry* entries, int* n_entries,
                               int* n_rows, int* pos, int* src) {
  __shared__ int s_rows[32], s_ents[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int i = tid; i < SK; i += blockDim.x) pos[i] = -1;
  for (int i = tid; i < R_max; i += blockDim.x) src[i] = -1;
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = tid * per, e1 = min(E, e0 + per);
  int rows = 0, ents = 0;
  for (int e = e0; e < e1; e++) {
    const int c = cnt[e];
    const int nch = (c + kPfRows - 1) / kPfRows;
    ents += nch;
    rows += nch > 0 ? (nch - 1) * kPfRows + ((c - (nch - 1) * kPfRows) + kPfPad - 1) / kPfPad * kPfPad : 0;
  }
  // exclusive block scan of (rows, ents)
  int ir = rows, ie = ents;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int r = __shfl_up_sync(0xffffffffu, ir, off), q = __shfl_up_sync(0xffffffffu, ie, off);
    if (lane >= off) {
      ir += r;
      ie += q;
    }
  }
  if (lane == 31) {
    s_rows[warp] = ir;
    s_ents[warp] = ie;
  }
  __syncthreads();
  int br = 0, be = 0, tr = 0, te = 0;
  for (int i = 0; i < nw; i++) {
    if (i < warp) {
      br += s_rows[i];
      be += s_ents[i];
    }
    tr += s_rows[i];
    te += s_ents[i];
  }
  int row = br + ir - rows, ent = be + ie - ents;
  for (int e = e0; e < e1; e++) {
    const int c = cnt[e];
    row_off[e] = row;
    for (int done = 0; done < c; done += kPfRows) {
      PfEntry en;
      en.e = e;
      en.row0 = row;
      en.n = min(kPfRows, c - done);
      en.npad = (en.n + kPfPad - 1) / kPfPad * kPfPad;
      entries[ent++] = en;
      row += en.npad;
    }
  }
  if (tid == 0) {
    *n_entries = te;
    *n_rows = tr;
  }
}

// One warp per expert: the grouped row of each of its routes (pos[t K + k]) and, per row, the token
// it holds (src; padding rows keep -1).
__global__ void pf_rank_kernel(const int32_t* idx, const int32_t* n_sel, int S, int K, int E, const int* cnt,
                               const int* row_off, int* pos, int* src) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (e >= E) return;
  const int c = cnt[e];
  if (c == 0) return;
  const int SK = S * K, row0 = row_off[e];
  int rank = 0;
  for (int base = 0; base < SK && rank < c; base += 32) {
    const bool m = pf_route_is(idx, n_sel, K, base + lane, SK, e);
    const unsigned bal = __ballot_sync(0xffffffffu, m);
    if (m) {
      const int row = row0 + rank + __popc(bal & ((1u << lane) - 1u));
      pos[base + lane] = row;
      src[row] = (base + lane) / K;
    }
    rank += __popc(bal);
  }
}

// One warp per grouped row: the token's activations in the tensor-core column order (each group of
// 8 columns as 0 4 1 5 2 6 3 7), or zeros for a padding row.
__global__ void pf_gather_kernel(const uint16_t* __restrict__ x, int D, int R_max, const int* n_rows, const int* src,
                                 uint16_t* __restrict__ xs) {
  const int lane = threadIdx.x & 31, G8 = D / 8;
  const int nr = *n_rows;
  for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < nr && row < R_max;
       row += gridDim.x * (blockDim.x >> 5)) {
    const int t = src[row];
    uint4* dr = reinterpret_cast<uint4*>(xs + (size_t)row * D);
    if (t < 0) {
      for (int g = lane; g < G8; g += 32) dr[g] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * D);
    for (int g = lane; g < G8; g += 32) {
      const uint4 v = __ldg(xr + g);  // columns 8g .. 8g+7 as bf16 pairs
      uint4 o;
      o.x = __byte_perm(v.x, v.z, 0x5410);  // (c0, c4)
      o.y = __byte_perm(v.x, v.z, 0x7632);  // (c1, c5)
      o.z = __byte_perm(v.y, v.w, 0x5410);  // (c2, c6)
      o.w = __byte_perm(v.y, v.w, 0x7632);  // (c3, c7)
      dr[g] = o;
    }
  }
}

// ------------------------------------------------------------------------------------------
// Dequantisation of packed int4 into the bf16 tensor-core layout
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));  // (a & mask) | bits
  return d;
}

// 8 nibbles (columns 8j .. 8j+7) -> 8 bf16 s (n - 8) in the order 0 4 1 5 2 6 3 7.
__device__ __forceinline__ uint4 pf_dequant8(uint32_t w, __nv_bfloat162 s2) {
  const __nv_bfloat162 c136 = __floats2bfloat162_rn(136.f, 136.f);
  uint32_t v[4];
  v[0] = lop3_and_or(w, 0x000f000fu, 0x43004300u);        // (128 + n0, 128 + n4)
  v[1] = lop3_and_or(w >> 4, 0x000f000fu, 0x43004300u);   // (n1, n5)
  v[2] = lop3_and_or(w >> 8, 0x000f000fu, 0x43004300u);   // (n2, n6)
  v[3] = lop3_and_or(w >> 12, 0x000f000fu, 0x43004300u);  // (n3, n7)
  uint4 o;
  uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v[i]);
    b = __hmul2(__hsub2(b, c136), s2);  // exact n - 8, then one rounding of the product
    op[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return o;
}

// ------------------------------------------------------------------------------------------
// Grouped GEMM with the tensor cores: DUAL = gate and up (epilogue SiLU(g) u -> bf16 h rows), else
// down (epilogue f32 rows of the routed outputs).
//   warp 0: TMA producer; warp 1: tensor-memory owner and MMA issuer; warps 2..9: converters;
//   warps 4..7 also read the accumulators (warp w reads tensor-memory lanes 32 (w % 4) ..).
// Work units are (entry, 128-row weight tile), strided over the persistent grid.
// ------------------------------------------------------------------------------------------

struct PfGemmParams {
  const ExpertDesc* table;
  const PfEntry* entries;
  const int* n_entries;
  int tiles;   // weight row tiles per entry: ceil(rows / 128)
  int rows;    // weight rows (I for gate/up, D for down)
  int K;       // reduction length (D for gate/up, I for down)
  int t0, t1;  // tensor indices in the expert descriptor (t1 < 0: single)
  void* out;   // DUAL: bf16 h [rows_total x rows] ; else f32 yr [rows_total x rows]
  int* err;
};

template <bool DUAL>
struct PfLayout {
  static constexpr int kT = DUAL ? 2 : 1;
  static constexpr uint32_t kA = 0;                                // kT bf16 weight tiles
  static constexpr uint32_t kAct = kT * kPfTileBytes;             // activation tile (<= 128 rows)
  static constexpr uint32_t kPacked = kAct + kPfTileBytes;        // kT packed tiles
  static constexpr uint32_t kStage = kPacked + kT * kPfPackedBytes;
  static constexpr uint32_t kAccCols = kT * 128;  // tensor-memory columns of one accumulator buffer
  static constexpr uint32_t kTmemCols = 2 * kAccCols;
  static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
};

struct PfCtrl {
  uint64_t full[kPfStages];   // TMA bytes of the stage landed
  uint64_t conv[kPfStages];   // converter warps wrote the stage's bf16 weight tiles
  uint64_t freed[kPfStages];  // the MMAs reading the stage completed
  uint64_t acc_full[2];       // accumulator buffer complete
  uint64_t acc_empty[2];      // accumulator buffer drained by the epilogue warps
  uint64_t mma_done;          // every MMA of this CTA completed (teardown)
  uint32_t tmem_base;
  int stop;
};

template <bool DUAL>
inline size_t pf_smem_bytes() {
  return 1024 + 1024 + (size_t)kPfStages * PfLayout<DUAL>::kStage;
}

__device__ __forceinline__ float pf_scale(const float* s, int gs, int G, int row, int col) {
  if (gs == 0) return __ldg(s + row);
  return __ldg(s + (size_t)row * G + col / gs);
}

__device__ __forceinline__ bool pf_wait(PfCtrl& c, uint64_t* bar, uint32_t parity, int* err) {
  if (ld_volatile_int(&c.stop)) return false;
  if (mbar_wait(bar, parity)) return true;
  set_error(err, COLI_E_TIMEOUT);
  *reinterpret_cast<volatile int*>(&c.stop) = 1;
  return false;
}

template <bool DUAL>
__global__ void __launch_bounds__(kPfThreads, 1) pf_gemm_kernel(PfGemmParams P, const __grid_constant__ CUtensorMap act_map) {
  using Lay = PfLayout<DUAL>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  PfCtrl& c = *reinterpret_cast<PfCtrl*>(base);
  uint8_t* stages = base + 1024;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < kPfStages; s++) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.conv[s], kPfConvWarps);
      mbar_init(&c.freed[s], 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&c.acc_full[b], 1);
      mbar_init(&c.acc_empty[b], 4);
    }
    mbar_init(&c.mma_done, 1);
    c.stop = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(&c.tmem_base, Lay::kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = c.tmem_base;

  const int n_units = *P.n_entries * P.tiles;
  const int nkt = (P.K + kPfKTile - 1) / kPfKTile;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (int u = blockIdx.x; u < n_units && !ld_volatile_int(&c.stop); u += gridDim.x) {
        const PfEntry en = P.entries[u / P.tiles];
        const int t = u % P.tiles;
        const ExpertDesc& ed = P.table[en.e];
        for (int kt = 0; kt < nkt; kt++) {
          if (!pf_wait(c, &c.freed[stage], phase ^ 1u, P.err)) break;
          uint8_t* st = stages + (size_t)stage * Lay::kStage;
          mbar_arrive_expect_tx(&c.full[stage], Lay::kT * kPfPackedBytes + (uint32_t)en.npad * 128u);
          tma_load_2d(st + Lay::kPacked, &ed.t[P.t0].map_tc, kt * kTcWords, t * kTcRows, &c.full[stage]);
          if (DUAL)
            tma_load_2d(st + Lay::kPacked + kPfPackedBytes, &ed.t[P.t1].map_tc, kt * kTcWords, t * kTcRows, &c.full[stage]);
          for (int j = 0; j < en.npad; j += 16)
            tma_load_2d(st + Lay::kAct + (uint32_t)j * 128u, &act_map, kt * kPfKTile, en.row0 + j, &c.full[stage]);
          issued++;
          if (++stage == kPfStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // after a timeout elsewhere, never leave with copies in flight: wait (bounded) for the last
      // issued phase of every stage
      if (ld_volatile_int(&c.stop))
        for (long long q = issued > kPfStages ? issued - kPfStages : 0; q < issued; q++)
          (void)mbar_wait(&c.full[q % kPfStages], (uint32_t)((q / kPfStages) & 1));
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int lu = 0;
      for (int u = blockIdx.x; u < n_units && !ld_volatile_int(&c.stop); u += gridDim.x, lu++) {
        const PfEntry en = P.entries[u / P.tiles];
        const int buf = lu & 1;
        const uint32_t idesc = bf16_f32_idesc(128, (uint32_t)en.npad);
        if (!pf_wait(c, &c.acc_empty[buf], (((uint32_t)lu >> 1) & 1u) ^ 1u, P.err)) break;
        tc_fence_after_sync();
        bool ok = true;
        for (int kt = 0; kt < nkt; kt++) {
          if (!pf_wait(c, &c.full[stage], phase, P.err) || !pf_wait(c, &c.conv[stage], phase, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          uint8_t* st = stages + (size_t)stage * Lay::kStage;
          const uint64_t bdesc = sw128_kmajor_desc(st + Lay::kAct);
#pragma unroll
          for (int x = 0; x < Lay::kT; x++) {
            const uint64_t adesc = sw128_kmajor_desc(st + Lay::kA + x * kPfTileBytes);
            const uint32_t dcol = tmem + (uint32_t)buf * Lay::kAccCols + (uint32_t)(x * 128);
#pragma unroll
            for (int ks = 0; ks < kPfKTile / 16; ks++)
              tc_mma_bf16(dcol, adesc + 2 * ks, bdesc + 2 * ks, idesc, kt > 0 || ks > 0);
          }
          tc_commit(&c.freed[stage]);
          if (++stage == kPfStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&c.acc_full[buf]);
      }
      tc_commit(&c.mma_done);  // teardown: tensor memory is released only after every MMA
      if (!mbar_wait(&c.mma_done, 0)) set_error(P.err, COLI_E_TIMEOUT);
    }
  } else {
    // ---------------- converters (+ epilogue on warps 4..7) ----------------
    const int cw = warp - 2;                 // converter warp 0..7
    const int ct = cw * 32 + lane;           // converter thread 0..255
    // DUAL: thread ct converts all 8 words of row ct % 128 of tensor ct / 128.
    // single: thread ct converts words 4 h .. 4 h + 3 (h = ct / 128) of row ct % 128.
    const int r = ct & (kTcRows - 1);
    const int x = DUAL ? (ct >> 7) : 0;
    const int w0 = DUAL ? 0 : (ct >> 7) * 4;
    constexpr int kW = DUAL ? 8 : 4;
    const bool epi = warp >= 4 && warp < 8;
    const int q = warp & 3;                  // tensor-memory lane quarter of an epilogue warp
    int stage = 0;
    uint32_t phase = 0;
    int lu = 0;
    for (int u = blockIdx.x; u < n_units && !ld_volatile_int(&c.stop); u += gridDim.x, lu++) {
      const PfEntry en = P.entries[u / P.tiles];
      const int t = u % P.tiles;
      const TensorDesc& td = P.table[en.e].t[x == 0 ? P.t0 : P.t1];
      const float* sp = td.s;
      const int gs = td.gs, G = td.G;
      const int row = t * kTcRows + r;
      const bool row_ok = row < P.rows;
      bool ok = true;
      for (int kt = 0; kt < nkt; kt++) {
        if (!pf_wait(c, &c.full[stage], phase, P.err)) {
          ok = false;
          break;
        }
        uint8_t* st = stages + (size_t)stage * Lay::kStage;
        const uint32_t* pk = reinterpret_cast<const uint32_t*>(st + Lay::kPacked + x * kPfPackedBytes + r * (kTcWords * 4));
        uint8_t* arow = st + Lay::kA + x * kPfTileBytes + r * 128;
        const int c0 = kt * kPfKTile;
        __nv_bfloat162 s_lo = __floats2bfloat162_rn(0.f, 0.f), s_hi = s_lo;
        if (row_ok) {
          const float a = c0 < P.K ? pf_scale(sp, gs, G, row, c0) : 0.f;
          const float b = c0 + 32 < P.K ? pf_scale(sp, gs, G, row, c0 + 32) : 0.f;
          s_lo = __floats2bfloat162_rn(a, a);
          s_hi = __floats2bfloat162_rn(b, b);
        }
#pragma unroll
        for (int j = 0; j < kW; j++) {
          const int wj = w0 + j;
          uint4 o = make_uint4(0, 0, 0, 0);
          if (row_ok && c0 + 8 * wj < P.K) o = pf_dequant8(pk[wj], wj < 4 ? s_lo : s_hi);
          *reinterpret_cast<uint4*>(arow + ((wj ^ (r & 7)) << 4)) = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.conv[stage]);
        if (++stage == kPfStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (epi) {
        // ---------------- epilogue of this unit ----------------
        const int buf = lu & 1;
        if (!pf_wait(c, &c.acc_full[buf], ((uint32_t)lu >> 1) & 1u, P.err)) break;
        tc_fence_after_sync();
        const int orow = t * kTcRows + q * 32 + lane;  // weight row this lane holds
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)buf * Lay::kAccCols;
        for (int n0 = 0; n0 < en.npad; n0 += 16) {
          float a[16];
          tmem_ld16(tl + (uint32_t)n0, a);
          if (DUAL) {
            float b[16];
            tmem_ld16(tl + 128u + (uint32_t)n0, b);
            if (orow < P.rows) {
              uint16_t* h = static_cast<uint16_t*>(P.out);
              const int pcol = (orow & ~7) + pf_perm8(orow & 7);
#pragma unroll
              for (int j = 0; j < 16; j++) {
                const int n = n0 + j;
                float v = 0.f;
                if (n < en.n) v = a[j] / (1.f + expf(-a[j])) * b[j];
                h[(size_t)(en.row0 + n) * P.rows + pcol] = f32_to_bf16_rn(v);
              }
            }
          } else if (orow < P.rows) {
            float* yr = static_cast<float*>(P.out);
#pragma unroll
            for (int j = 0; j < 16; j++)
              if (n0 + j < en.n) yr[(size_t)(en.row0 + n0 + j) * P.rows + orow] = a[j];
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.acc_empty[buf]);
      }
    }
  }
  // teardown: every role is out of its loop; the MMA issuer has seen its last MMA complete
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, Lay::kTmemCols);
}

// ------------------------------------------------------------------------------------------
// Combine: y[t] = resid[t] + sum over kept slots k (in slot order) of w[t, k] yr[pos[t, k]].
// ------------------------------------------------------------------------------------------

__global__ void pf_combine_kernel(const float* __restrict__ yr, const int* __restrict__ pos, const float* __restrict__ w,
                                  const int32_t* __restrict__ n_sel, int S, int K, int D, const void* resid, int dtype,
                                  void* y, int* err) {
  const long long n = (long long)S * D;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / D), d = (int)(i - (long long)t * D);
    int ns = n_sel ? __ldg(n_sel + t) : K;
    ns = ns < 0 ? 0 : (ns > K ? K : ns);
    float acc = 0.f;
    for (int k = 0; k < ns; k++) {
      const int p = __ldg(pos + t * K + k);
      if (p < 0) {
        if (d == 0) set_error(err, COLI_E_ROUTE);
        continue;
      }
      acc = fmaf(__ldg(w + t * K + k), __ldg(yr + (size_t)p * D + d), acc);
    }
    if (resid) acc = load_act(resid, dtype, (size_t)t * D + d) + acc;
    if (dtype == COLI_DTYPE_F32)
      static_cast<float*>(y)[(size_t)t * D + d] = acc;
    else
      static_cast<uint16_t*>(y)[(size_t)t * D + d] = f32_to_bf16_rn(acc);
  }
}

// ------------------------------------------------------------------------------------------
// Host launcher
// ------------------------------------------------------------------------------------------

// bf16 activations (16-byte-aligned rows); D and I multiples of 8; every expert's group size 0 or a multiple of 32; on
// average at least kPfMinRows routed rows per expert of the table.
constexpr int kPfMinRows = 8;
bool prefill_eligible(const coli_ctx* ctx, const void* x, int S, int K, int x_dtype) {
  if (x_dtype != COLI_DTYPE_BF16 || (reinterpret_cast<uintptr_t>(x) & 15) != 0 || ctx->table_D % 8 != 0 || ctx->table_I % 8 != 0 || ctx->table_count == 0) return false;
  if ((long long)S * K < (long long)kPfMinRows * ctx->table_count) return false;
  for (int e = 0; e < COLI_MAX_EXPERTS; e++) {
    const ExpertDesc& d = ctx->h_table[e];
    if (!d.valid) continue;
    for (int t = 0; t < 3; t++)
      if (d.t[t].gs != 0 && d.t[t].gs % 32 != 0) return false;
  }
  return true;
}

int launch_prefill(coli_ctx* ctx, const void* x, int S, const int32_t* idx, const float* w, const int32_t* n_sel,
                   int K, const void* resid, void* y) {
  const int D = ctx->table_D, I = ctx->table_I;
  int E = 0, n_valid = 0;
  for (int e = 0; e < COLI_MAX_EXPERTS; e++)
    if (ctx->h_table[e].valid) {
      E = e + 1;
      n_valid++;
    }
  const long long SK = (long long)S * K;
  const long long R_max = SK + (long long)(kPfPad - 1) * n_valid + kPfPad;
  const long long max_entries = SK / kPfRows + n_valid + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t o_cnt = take((size_t)E * 4), o_roff = take((size_t)E * 4), o_nent = take(8),
               o_ent = take((size_t)max_entries * sizeof(PfEntry)), o_pos = take((size_t)SK * 4),
               o_src = take((size_t)R_max * 4),
               o_xs = take((size_t)R_max * D * 2), o_hs = take((size_t)R_max * I * 2), o_yr = take((size_t)R_max * D * 4);
  int rc = ensure_workspace(ctx, off);
  if (rc != COLI_OK) return rc;
  uint8_t* ws = reinterpret_cast<uint8_t*>(ctx->ws.base);
  int* cnt = reinterpret_cast<int*>(ws + o_cnt);
  int* roff = reinterpret_cast<int*>(ws + o_roff);
  int* nent = reinterpret_cast<int*>(ws + o_nent);
  PfEntry* ents = reinterpret_cast<PfEntry*>(ws + o_ent);
  int* pos = reinterpret_cast<int*>(ws + o_pos);
  int* src = reinterpret_cast<int*>(ws + o_src);
  int* nrows = nent + 1;
  uint16_t* xs = reinterpret_cast<uint16_t*>(ws + o_xs);
  uint16_t* hs = reinterpret_cast<uint16_t*>(ws + o_hs);
  float* yr = reinterpret_cast<float*>(ws + o_yr);

  CUtensorMap xs_map, hs_map;
  if ((rc = encode_bf16_rows_map(ctx, &xs_map, xs, R_max, D)) != COLI_OK) return rc;
  if ((rc = encode_bf16_rows_map(ctx, &hs_map, hs, R_max, I)) != COLI_OK) return rc;

  cudaError_t e;
  const int wpb = 8;  // warps (experts) per block of the grouping kernels
  pf_count_kernel<<<(E + wpb - 1) / wpb, wpb * 32, 0, ctx->stream>>>(idx, n_sel, S, K, E, ctx->d_table, cnt);
  pf_plan_kernel<<<1, 1024, 0, ctx->stream>>>(cnt, E, (int)SK, (int)R_max, roff, ents, nent, nrows, pos, src);
  pf_rank_kernel<<<(E + wpb - 1) / wpb, wpb * 32, 0, ctx->stream>>>(idx, n_sel, S, K, E, cnt, roff, pos, src);
  {
    int g = (int)((R_max + 7) / 8);
    if (g > 8 * ctx->num_sms) g = 8 * ctx->num_sms;
    pf_gather_kernel<<<g, 256, 0, ctx->stream>>>(static_cast<const uint16_t*>(x), D, (int)R_max, nrows, src, xs);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "prefill grouping launch");

  PfGemmParams G{};
  G.table = ctx->d_table;
  G.entries = ents;
  G.n_entries = nent;
  G.err = ctx->d_status;
  {
    const size_t smem = pf_smem_bytes<true>();
    if ((e = cudaFuncSetAttribute(pf_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return cuda_fail(ctx, e, "prefill gate/up smem attribute");
    G.tiles = (I + kTcRows - 1) / kTcRows;
    G.rows = I;
    G.K = D;
    G.t0 = T_GATE;
    G.t1 = T_UP;
    G.out = hs;
    ProfScope prof(ctx, COLI_KERNEL_GATEUP);
    pf_gemm_kernel<true><<<ctx->num_sms, kPfThreads, smem, ctx->stream>>>(G, xs_map);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "prefill gate/up launch");
  }
  {
    const size_t smem = pf_smem_bytes<false>();
    if ((e = cudaFuncSetAttribute(pf_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return cuda_fail(ctx, e, "prefill down smem attribute");
    G.tiles = (D + kTcRows - 1) / kTcRows;
    G.rows = D;
    G.K = I;
    G.t0 = T_DOWN;
    G.t1 = -1;
    G.out = yr;
    ProfScope prof(ctx, COLI_KERNEL_DOWN);
    pf_gemm_kernel<false><<<ctx->num_sms, kPfThreads, smem, ctx->stream>>>(G, hs_map);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "prefill down launch");
  }
  {
    const long long n = SK / K * D;
    int grid = (int)((n + 255) / 256);
    if (grid > 8 * ctx->num_sms) grid = 8 * ctx->num_sms;
    ProfScope prof(ctx, COLI_KERNEL_COMBINE);
    pf_combine_kernel<<<grid, 256, 0, ctx->stream>>>(yr, pos, w, n_sel, S, K, D, resid, COLI_DTYPE_BF16, y, ctx->d_status);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "prefill combine launch");
  }
  return COLI_OK;
}

}  // namespace coli
