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
// GEMM orientation. An expert's tokens are the MMA's M side (128 rows; rows past the entry's tokens
// are ignored) and a 256-row block of weights is its N side: the gate and the up tile of the same
// 128 rows, or two consecutive 128-row tiles of the down matrix. The accumulator D = X W^T sits in
// tensor memory with a token per lane and a weight row per column. Four MMAs of K = 16 cover a
// 64-column K tile whatever the number of tokens (the single issuing thread spends a roughly fixed
// time per MMA instruction, so fewer, wider instructions are what sets the K-tile rate).
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

#ifndef COLI_PF_ROWS
#define COLI_PF_ROWS 128
#endif
#ifndef COLI_PF_CONV_WARPS
#define COLI_PF_CONV_WARPS 16
#endif
constexpr int kPfRows = COLI_PF_ROWS;  // tokens (the MMA's M) per work entry
static_assert(kPfRows == 128, "the epilogue reads the accumulator in the M = 128 layout: a token per lane");
constexpr int kPfPad = 16;      // per-entry token blocks are padded to a multiple of 16
constexpr int kPfKTile = 64;    // K columns per pipeline stage
constexpr int kPfConvWarps = COLI_PF_CONV_WARPS;  // warps 3.. convert; warps 4..7 also drain the accumulator
constexpr int kPfThreads = (3 + kPfConvWarps) * 32;  // + the two producer warps and the MMA warp
static_assert(kPfThreads <= 1024, "one CTA holds every role");
constexpr uint32_t kPfTileBytes = kTcRows * 128;       // one bf16 operand tile: 128 rows x 128 bytes
constexpr uint32_t kPfPackedBytes = kTcRows * kTcWords * 4;  // one packed int4 weight tile (4 K tiles)
constexpr int kPfSuper = kTcWords * 8 / kPfKTile;            // K tiles per packed tile

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

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_splat(float f) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(f));
  return d;
}

constexpr uint32_t kBf16x2_136 = 0x43084308u;  // (136, 136): the magic 128 plus the offset 8

// 8 nibbles (columns 8j .. 8j+7) -> 8 bf16 values s (n - 8) in the order 0 4 1 5 2 6 3 7.
// (0x4300 | n) is the bf16 number 128 + n; subtracting 136 is exact, the product rounds once.
__device__ __forceinline__ uint4 pf_dequant8(uint32_t w, uint32_t s2) {
  uint4 o;
  o.x = bf16x2_mul(bf16x2_sub(lop3_and_or(w, 0x000f000fu, 0x43004300u), kBf16x2_136), s2);        // (n0, n4)
  o.y = bf16x2_mul(bf16x2_sub(lop3_and_or(w >> 4, 0x000f000fu, 0x43004300u), kBf16x2_136), s2);   // (n1, n5)
  o.z = bf16x2_mul(bf16x2_sub(lop3_and_or(w >> 8, 0x000f000fu, 0x43004300u), kBf16x2_136), s2);   // (n2, n6)
  o.w = bf16x2_mul(bf16x2_sub(lop3_and_or(w >> 12, 0x000f000fu, 0x43004300u), kBf16x2_136), s2);  // (n3, n7)
  return o;
}

// ------------------------------------------------------------------------------------------
// Grouped GEMM with the tensor cores: DUAL = gate and up (epilogue SiLU(g) u -> bf16 h rows), else
// down (epilogue f32 rows of the routed outputs). Three rings decouple the latencies:
//   packed ring (kPkStages): packed int4 tiles, staged by TMA far ahead of their use;
//   act ring (kActStages): 128-byte-swizzled bf16 activation tiles, staged by TMA;
//   operand ring (kOpStages): bf16 weight tiles written by the converter warps.
// A converter warp releases a packed stage only after the words it loaded from it are consumed (its
// dequantised stores done): released right after the shared-memory loads were issued, the copy engine
// could refill the stage before every load had read it, under the tensor core's operand traffic.
// warp 0 stages packed tiles; warp 1 owns tensor memory, its lane 0 issues the MMAs; warp 2 stages
// activation tiles (each producer has a warp of its own, so neither waits while the other sleeps
// in a barrier wait); warps 3.. convert; warps 4..7 also read the accumulators (warp w reads
// tensor-memory lanes 32 (w % 4) ..: tokens). Work units are (entry, 256-row weight block), strided over
// the persistent grid; every role walks the same units and K tiles.
// ------------------------------------------------------------------------------------------

#ifndef COLI_PF_PK_STAGES
#define COLI_PF_PK_STAGES 2
#endif
#ifndef COLI_PF_ACT_STAGES
#define COLI_PF_ACT_STAGES 3
#endif
#ifndef COLI_PF_OP_STAGES
#define COLI_PF_OP_STAGES 3
#endif
constexpr int kPkStages = COLI_PF_PK_STAGES;
constexpr int kActStages = COLI_PF_ACT_STAGES;
constexpr int kOpStages = COLI_PF_OP_STAGES;

struct PfGemmParams {
  const ExpertDesc* table;
  const PfEntry* entries;
  const int* n_entries;
  int tiles;   // 256-row weight blocks per entry: ceil(rows / 128) (DUAL) or ceil(rows / 256)
  int rows;    // weight rows (I for gate/up, D for down)
  int K;       // reduction length (D for gate/up, I for down)
  int t0, t1;  // tensor indices in the expert descriptor (t1 < 0: single)
  void* out;   // DUAL: bf16 h [rows_total x rows] ; else f32 yr [rows_total x rows]
  int* err;
};

template <bool DUAL>
struct PfLayout {
  static constexpr int kT = 2;  // 128-row weight tiles per block (the two halves of the MMA's N)
  static constexpr uint32_t kOpStage = kT * kPfTileBytes;            // bf16 weight tiles
  static constexpr uint32_t kActStage = kPfRows * 128;               // <= kPfRows rows x 128 bytes
  static constexpr uint32_t kPkStage = kT * kPfPackedBytes;          // packed tiles
  static constexpr uint32_t kOp = 0;
  static constexpr uint32_t kAct = kOp + kOpStages * kOpStage;
  static constexpr uint32_t kPk = kAct + kActStages * kActStage;
  static constexpr uint32_t kBytes = kPk + kPkStages * kPkStage;
  static_assert(kAct % 1024 == 0 && kPk % 1024 == 0 && kOpStage % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static constexpr uint32_t kAccCols = kT * kPfRows;  // tensor-memory columns of the accumulator
  static constexpr uint32_t kTmemCols = kAccCols;
};

struct PfCtrl {
  uint64_t pk_full[kPkStages], pk_empty[kPkStages];
  uint64_t act_full[kActStages], act_empty[kActStages];
  uint64_t op_full[kOpStages], op_empty[kOpStages];
  uint64_t acc_full;      // accumulator complete
  uint64_t acc_empty;     // accumulator drained by the epilogue warps
  uint64_t mma_done;      // every MMA of this CTA completed (teardown)
  uint32_t tmem_base;
  int stop;
};
static_assert(sizeof(PfCtrl) <= 1024, "control block");

template <bool DUAL>
inline size_t pf_smem_bytes() {
  return 1024 + 1024 + PfLayout<DUAL>::kBytes;
}

__device__ __forceinline__ bool pf_wait(PfCtrl& c, uint64_t* bar, uint32_t parity, int* err) {
  if (ld_volatile_int(&c.stop)) return false;
  if (mbar_wait(bar, parity)) return true;
  set_error(err, COLI_E_TIMEOUT);
  *reinterpret_cast<volatile int*>(&c.stop) = 1;
  return false;
}

// ring position: stage index and phase parity, advanced once per K tile
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

template <bool DUAL>
__global__ void __launch_bounds__(kPfThreads, 1) pf_gemm_kernel(PfGemmParams P, const __grid_constant__ CUtensorMap act_map) {
  using Lay = PfLayout<DUAL>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  PfCtrl& c = *reinterpret_cast<PfCtrl*>(base);
  uint8_t* sm = base + 1024;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < kPkStages; s++) {
      mbar_init(&c.pk_full[s], 1);
      mbar_init(&c.pk_empty[s], kPfConvWarps);
    }
    for (int s = 0; s < kActStages; s++) {
      mbar_init(&c.act_full[s], 1);
      mbar_init(&c.act_empty[s], 1);
    }
    for (int s = 0; s < kOpStages; s++) {
      mbar_init(&c.op_full[s], kPfConvWarps);
      mbar_init(&c.op_empty[s], 1);
    }
    mbar_init(&c.acc_full, 1);
    mbar_init(&c.acc_empty, 4);
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

  if ((warp == 0 || warp == 2) && lane == 0) {
    // ---------------- TMA producers: warp 0 packed tiles, warp 2 activation tiles ----------------
    const bool packed = warp == 0;
    const int nst = packed ? kPkStages : kActStages;
    uint64_t* fullb = packed ? c.pk_full : c.act_full;
    uint64_t* emptyb = packed ? c.pk_empty : c.act_empty;
    RingPos rp;
    long long issued = 0;
    // weights stream through L2 once; the grouped activation rows are read by every weight tile of
    // their entry, so they are kept in L2 ahead of the weights
    const uint64_t policy = packed ? l2_evict_first_policy() : l2_evict_last_policy();
    for (int u = blockIdx.x; u < n_units && !ld_volatile_int(&c.stop); u += gridDim.x) {
      const PfEntry en = P.entries[u / P.tiles];
      const int t = u % P.tiles;
      const ExpertDesc& ed = P.table[en.e];
      for (int kt = 0; kt < nkt; kt++) {
        if (packed && kt % kPfSuper != 0) continue;  // one packed tile covers kPfSuper K tiles
        if (!pf_wait(c, &emptyb[rp.s], rp.ph ^ 1u, P.err)) break;
        if (packed) {
          uint8_t* st = sm + Lay::kPk + (size_t)rp.s * Lay::kPkStage;
          // the second tile of a down block may lie wholly past the last row: TMA fills it with
          // zeros and still delivers its bytes
          mbar_arrive_expect_tx(&fullb[rp.s], Lay::kPkStage);
          const int kx = (kt / kPfSuper) * kTcWords;
          tma_load_2d_hint(st, &ed.t[P.t0].map_tc, kx, (DUAL ? t : 2 * t) * kTcRows, &fullb[rp.s], policy);
          tma_load_2d_hint(st + kPfPackedBytes, &ed.t[DUAL ? P.t1 : P.t0].map_tc, kx, (DUAL ? t : 2 * t + 1) * kTcRows,
                           &fullb[rp.s], policy);
        } else {
          uint8_t* st = sm + Lay::kAct + (size_t)rp.s * Lay::kActStage;
          mbar_arrive_expect_tx(&fullb[rp.s], (uint32_t)en.npad * 128u);
          for (int j = 0; j < en.npad; j += 16)
            tma_load_2d_hint(st + (uint32_t)j * 128u, &act_map, kt * kPfKTile, en.row0 + j, &fullb[rp.s], policy);
        }
        issued++;
        rp.next(nst);
      }
    }
    // after a timeout elsewhere, never leave with copies in flight: wait (bounded) for the last
    // issued phase of every stage
    if (ld_volatile_int(&c.stop))
      for (long long q = issued > nst ? issued - nst : 0; q < issued; q++)
        (void)mbar_wait(&fullb[q % nst], (uint32_t)((q / nst) & 1));
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      RingPos ra, ro;
      int lu = 0;
      for (int u = blockIdx.x; u < n_units && !ld_volatile_int(&c.stop); u += gridDim.x, lu++) {
        const uint32_t idesc = bf16_f32_idesc(kPfRows, Lay::kT * kTcRows);  // M = tokens, N = weight rows
        if (!pf_wait(c, &c.acc_empty, ((uint32_t)lu & 1u) ^ 1u, P.err)) break;
        tc_fence_after_sync();
        bool ok = true;
        for (int kt = 0; kt < nkt; kt++) {
          if (!pf_wait(c, &c.act_full[ra.s], ra.ph, P.err) || !pf_wait(c, &c.op_full[ro.s], ro.ph, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = sw128_kmajor_desc(sm + Lay::kAct + (size_t)ra.s * Lay::kActStage);
          const uint64_t bdesc = sw128_kmajor_desc(sm + Lay::kOp + (size_t)ro.s * Lay::kOpStage);  // both tiles
#pragma unroll
          for (int ks = 0; ks < kPfKTile / 16; ks++)
            tc_mma_bf16(tmem, adesc + 2 * ks, bdesc + 2 * ks, idesc, kt > 0 || ks > 0);
          tc_commit(&c.act_empty[ra.s]);
          tc_commit(&c.op_empty[ro.s]);
          ra.next(kActStages);
          ro.next(kOpStages);
        }
        if (!ok) break;
        tc_commit(&c.acc_full);
      }
      tc_commit(&c.mma_done);  // teardown: tensor memory is released only after every MMA
      if (!mbar_wait(&c.mma_done, 0)) set_error(P.err, COLI_E_TIMEOUT);
    }
  } else if (warp >= 3) {
    // ---------------- converters (+ epilogue on warps 4..7) ----------------
    const int ct = (warp - 3) * 32 + lane;   // converter thread 0..511
    // kParts threads share a row of a tensor: thread ct converts words w0 .. w0 + kW - 1 (w0 = kW
    // ((ct / 128) % kParts)) of row ct % 128 of tensor ct / (128 kParts).
    constexpr int kParts = kPfConvWarps * 32 / (Lay::kT * kTcRows);
    constexpr int kW = 8 / kParts;  // words of a 64-column K tile (8 words per row) per thread
    static_assert(kParts * kW == 8 && kW >= 2, "converter split");
    static_assert(kW <= 4, "a thread's columns of a K tile must lie in one 32-column part (one scale)");
    const int r = ct & (kTcRows - 1);
    const int x = ct / (kTcRows * kParts);   // weight tile of the block
    const int w0 = ((ct / kTcRows) % kParts) * kW;
    const bool epi = warp >= 4 && warp < 8;
    const int q = warp & 3;                  // tensor-memory lane quarter of an epilogue warp
    const uint32_t swz = (uint32_t)(r & 7);
    RingPos rp, ro;
    int lu = 0;
    for (int u = blockIdx.x; u < n_units && !ld_volatile_int(&c.stop); u += gridDim.x, lu++) {
      const PfEntry en = P.entries[u / P.tiles];
      const int t = u % P.tiles;
      const TensorDesc& td = P.table[en.e].t[(DUAL && x == 1) ? P.t1 : P.t0];
      const int gs = td.gs, row = (DUAL ? t : 2 * t + x) * kTcRows + r;
      const bool row_ok = row < P.rows;
      const float* srow = row_ok ? td.s + (gs == 0 ? (size_t)row : (size_t)row * td.G) : nullptr;
      // this thread's 32-column half of every K tile: columns c0 + 8 w0 .. + 8 kW - 1 (gs is 0 or a
      // multiple of 32, so the half has one scale); its group advances incrementally
      const int hoff = 8 * w0;
      int grp = 0, nb = gs > 0 ? gs : 0;
      auto scale_of = [&](int col) -> float {
        if (!row_ok || col >= P.K) return 0.f;
        if (gs == 0) return __ldg(srow);
        while (col >= nb) {
          grp++;
          nb += gs;
        }
        return __ldg(srow + grp);
      };
      float s_next0 = scale_of(hoff), s_next1 = nkt > 1 ? scale_of(kPfKTile + hoff) : 0.f;  // two K tiles ahead
      bool ok = true;
      for (int kt = 0; kt < nkt; kt++) {
        const uint32_t s2 = bf16x2_splat(s_next0);
        s_next0 = s_next1;
        s_next1 = kt + 2 < nkt ? scale_of((kt + 2) * kPfKTile + hoff) : 0.f;
        const int sub = kt % kPfSuper;  // K tile within the packed tile
        if ((sub == 0 && !pf_wait(c, &c.pk_full[rp.s], rp.ph, P.err)) ||
            !pf_wait(c, &c.op_empty[ro.s], ro.ph ^ 1u, P.err)) {
          ok = false;
          break;
        }
        // row r of the packed tile is 128 bytes, its 16-byte chunks swizzled by r % 8 (TMA 128B mode);
        // this thread's words are bytes 4 (8 sub + w0) .. of the row
        const uint8_t* prow = sm + Lay::kPk + (size_t)rp.s * Lay::kPkStage + x * kPfPackedBytes + r * 128;
        auto pk_at = [&](int word) {  // address of word `word` (0..31) of this row
          const uint32_t b = 4u * (uint32_t)word;
          return prow + ((((b >> 4) ^ swz) << 4) | (b & 15u));
        };
        uint8_t* arow = sm + Lay::kOp + (size_t)ro.s * Lay::kOpStage + x * kPfTileBytes + r * 128;
        uint32_t wv[kW];
        if (kW >= 4) {
#pragma unroll
          for (int j = 0; j < kW; j += 4) {
            const uint4 v = lds128(pk_at(8 * sub + w0 + j));  // 4 words in one 16-byte chunk
            wv[j] = v.x;
            wv[(j + 1) % kW] = v.y;
            wv[(j + 2) % kW] = v.z;
            wv[(j + 3) % kW] = v.w;
          }
        } else {
          uint2 v;
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(pk_at(8 * sub + w0))) : "memory");
          wv[0] = v.x;
          wv[kW - 1] = v.y;
        }
        const bool last_sub = sub == kPfSuper - 1 || kt + 1 == nkt;
        const int c0 = kt * kPfKTile + hoff;
        if (row_ok && c0 + 8 * kW <= P.K) {  // whole half inside the matrix
#pragma unroll
          for (int j = 0; j < kW; j++)
            *reinterpret_cast<uint4*>(arow + (((uint32_t)(w0 + j) ^ swz) << 4)) = pf_dequant8(wv[j], s2);
        } else {
#pragma unroll
          for (int j = 0; j < kW; j++) {
            uint4 o = make_uint4(0, 0, 0, 0);
            if (row_ok && c0 + 8 * j < P.K) o = pf_dequant8(wv[j], s2);
            *reinterpret_cast<uint4*>(arow + (((uint32_t)(w0 + j) ^ swz) << 4)) = o;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (last_sub) mbar_arrive(&c.pk_empty[rp.s]);  // the packed words are consumed
          mbar_arrive(&c.op_full[ro.s]);
        }
        if (last_sub) rp.next(kPkStages);
        ro.next(kOpStages);
      }
      if (!ok) break;
      if (epi) {
        // ---------------- epilogue of this unit: lane = token, column = weight row ----------------
        if (!pf_wait(c, &c.acc_full, (uint32_t)lu & 1u, P.err)) break;
        tc_fence_after_sync();
        const int m = q * 32 + lane;  // token of the entry this lane holds
        const bool tok = m < en.n;
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        if (DUAL) {
          // h = SiLU(g) u for weight rows i of the tile, stored in the tensor-core column order:
          // within each group of 8, word p holds columns p and p + 4
          uint16_t* hrow = static_cast<uint16_t*>(P.out) + (size_t)(en.row0 + m) * P.rows;
          for (int j0 = 0; j0 < kTcRows; j0 += 16) {
            float g[16], uu[16];
            tmem_ld16(tl + (uint32_t)j0, g);
            tmem_ld16(tl + (uint32_t)(kTcRows + j0), uu);
#pragma unroll
            for (int half = 0; half < 2; half++) {
              const int i8 = t * kTcRows + j0 + 8 * half;
              if (!tok || i8 >= P.rows) continue;
              uint32_t wv[4];
#pragma unroll
              for (int p = 0; p < 4; p++) {
                const float a0 = g[8 * half + p], a1 = g[8 * half + p + 4];
                const float v0 = a0 / (1.f + expf(-a0)) * uu[8 * half + p];
                const float v1 = a1 / (1.f + expf(-a1)) * uu[8 * half + p + 4];
                wv[p] = (uint32_t)f32_to_bf16_rn(v0) | ((uint32_t)f32_to_bf16_rn(v1) << 16);
              }
              *reinterpret_cast<uint4*>(hrow + i8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
        } else {
          float* yrow = static_cast<float*>(P.out) + (size_t)(en.row0 + m) * P.rows;
          for (int j0 = 0; j0 < Lay::kT * kTcRows; j0 += 16) {
            float a[16];
            tmem_ld16(tl + (uint32_t)j0, a);
            const int d0 = 2 * t * kTcRows + j0;
#pragma unroll
            for (int v = 0; v < 4; v++)
              if (tok && d0 + 4 * v < P.rows)
                *reinterpret_cast<float4*>(yrow + d0 + 4 * v) = make_float4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.acc_empty);
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
                                  void* y, int y_dtype, int* err) {
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
    if (y_dtype == COLI_DTYPE_F32)
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
                   int K, const void* resid, void* y, int y_dtype) {
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
    G.tiles = (D + 2 * kTcRows - 1) / (2 * kTcRows);
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
    pf_combine_kernel<<<grid, 256, 0, ctx->stream>>>(yr, pos, w, n_sel, S, K, D, resid, COLI_DTYPE_BF16, y, y_dtype,
                                                     ctx->d_status);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(ctx, e, "prefill combine launch");
  }
  return COLI_OK;
}

}  // namespace coli
