// S = 1 decode: the whole grouped int4 expert FFN of one token -- gate + up dual GEMV, SiLU(g) * u,
// the down GEMV, per-expert weighting and a fixed-order reduce into the residual -- as one persistent
// streaming kernel that reads every kept expert's weights once, and a small reduce kernel.
//
// Sources: c/backend_cuda.cu commit history, commit "The TC_W4A16 branch ..." (the grouped decode
// path: dual gate/up GEMV, SiLU, down GEMV), commit "grouped MoE kernels were per-row-only" (per-row
// and per-group scales, mixed members in one launch); PR #434 "COLI_CUDA_RESID=1", section "What"
// (per-expert weighting and a fixed-order reduce on the device, no atomics).
//
// Work split. The hidden dimension I of every kept slot is cut into units of kPanelCols (16) rows.
// A unit's gate and up rows give 16 values of h = SiLU(g) u, and those are all the down projection
// needs from the unit: y_k[d] receives sum over the unit's i of Wd[d, i] h_i. So a CTA streams, for
// each of its units, the 16 gate rows, the 16 up rows and the same 16 columns of down (kept
// panel-major by the library, one contiguous [D x 8 byte] block per unit), and adds
// w_k * scale * (the unit's down dot product) into its own partial row of y. No CTA waits for
// another CTA, so each CTA's weight stream runs from its first unit to its last without a
// dependency bubble. Every CTA stores its partial row; the reduce kernel, chained by programmatic
// dependent launch, adds the partial rows in CTA order and then the residual: a fixed-order,
// atomics-free reduce, bit-identical from run to run.
//
// Roles inside a CTA (D = 512 NW, NW consumer warps per role):
//   - NW gate/up warps: one 32-column chunk of x per thread (its limbs in registers), two thread
//     rows; per unit they dot the 16 gate and 16 up rows with x and leave each warp's row sums;
//   - one warp that turns a unit's row sums into h = SiLU(g s_g) (u s_u) and its limbs;
//   - NW down warps: 16 rows of y per thread; per unit they dot the unit's down panel with h and
//     accumulate w_k s_d times that into their rows of the partial;
//   - two producer lanes that fill a gate/up ring and a down ring of shared-memory stages with bulk
//     asynchronous copies (cp.async.bulk, completion on mbarriers).
// The gate/up warps run ahead of the down warps by up to kHB units (the row sums and h limbs are
// kHB-deep rings with back-pressure), so a unit's down work overlaps the next units' gate/up work on
// other warps. Every wait is bounded and suspends in mbarrier.try_wait.
//
// Arithmetic: the block-fixed-point dp4a dot product of dot.h. Gate and up use 32-column chunks of
// x; the down projection uses the unit's 16 values of h as one 16-column block (its own power-of-two
// scale), so each down dot product has the same error bound as a chunk of the gate/up ones.
#include "coli_internal.h"
#include "dot.h"
#include "pipe.h"

namespace coli {

constexpr int kStMaxStages = 4;   // per ring
constexpr int kStMaxWarps = 12;   // warps per consumer role: D <= 6144 (two stages of each ring fit)
constexpr int kHB = 4;            // units of row sums and h limbs in flight between the roles

struct StreamSlot {
  const uint8_t* gw;  // gate rows [I x D/2]
  const uint8_t* uw;  // up rows [I x D/2]
  const uint8_t* dp;  // down panels [I/16][D][8 bytes]
  const float* gs;    // gate scales: [I] (per row) or [I x Gg] (chunk groups)
  const float* us;    // up scales
  const float* ds;    // down scales: [D] (per row) or transposed chunk-group scales [Gd x D]
  float wk;           // routing weight of the slot
  int gmode, umode, dmode;
  int Gg, Gu;         // scales per gate / up row (1 per row, or one per chunk group)
  int gsg, gsu, gsd;  // group sizes (0: per row)
  int ok;
};

struct StreamCtrl {
  uint64_t full_g[kStMaxStages], empty_g[kStMaxStages];  // gate/up ring
  uint64_t full_d[kStMaxStages], empty_d[kStMaxStages];  // down ring
  uint64_t redf[kHB], redfree[kHB];  // row sums of unit n stored (buffer n % kHB) / read by the h warp
  uint64_t hlf[kHB], hlfree[kHB];    // h limbs of unit n stored / read by every down warp
  StreamSlot slot[COLI_MAX_K];
  float red[kHB][kStMaxWarps][16];   // per gate/up warp: its 8 gate and 8 up row sums of a unit
  float fs[kHB][2][16];              // per-row gate and up scales of a unit's 16 rows (1 for chunk scales)
  Limbs16 hl[kHB];                   // h of a unit as one 16-column block of limbs
  uint64_t xfull, xfree;             // x copied into gate/up stage 0 / every gate/up warp has read it
  int m;
};

struct StreamParams {
  const void* x;
  int x_dtype;
  int D, I, K;
  const int32_t* idx;
  const float* w;
  const int32_t* n_sel;
  const ExpertDesc* table;
  float* part;               // [gridDim.x x D] partial rows
  int* err;
  int nsg, nsd;              // stages of the gate/up ring and of the down ring
  uint32_t sbg, sbd;         // their stage bytes
  unsigned long long wait_ns;
  int withhold;              // test hook: the CTA owning unit 0 withholds the copy of its first gate stage
  int x_bulk;                // x is 16-byte aligned: each CTA copies it whole into shared memory
};

// Limbs of 16 values of h held by lanes 0..15 (lanes 16..31 hold 0); every lane returns the same
// limbs: lane 8 w + 2 b + p holds column 8 w + 2 b + p, whose digits go to byte b of word (w, p).
__device__ __forceinline__ bool warp_limbs16(float h, int lane, Limbs16& L) {
  float M = fabsf(h);
  const bool bad = !(fmaf(h, 0.f, 0.f) == 0.f);  // NaN or infinite
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const bool finite = !__any_sync(0xffffffffu, bad);
  int e = 0;
  if (finite && M > 0.f) frexpf(M, &e);  // M < 2^e
  int q = 22 - e;                         // M 2^q in [2^21, 2^22)
  q = q > 122 ? 122 : q;
  const float scale = (finite && M > 0.f) ? __int_as_float((127 + q) << 23) : 0.f;
  const int xi = __float2int_rn(h * scale);
  const uint32_t z = ((uint32_t)xi + 0x808080u) ^ 0x808080u;
#pragma unroll
  for (int w = 0; w < 2; w++)
#pragma unroll
    for (int p = 0; p < 2; p++) {
      const uint32_t z0 = __shfl_sync(0xffffffffu, z, 8 * w + p), z1 = __shfl_sync(0xffffffffu, z, 8 * w + 2 + p);
      const uint32_t z2 = __shfl_sync(0xffffffffu, z, 8 * w + 4 + p), z3 = __shfl_sync(0xffffffffu, z, 8 * w + 6 + p);
      const uint32_t a01 = prmt(z0, z1, 0x5140u), a23 = prmt(z2, z3, 0x5140u);
      const uint32_t c01 = prmt(z0, z1, 0x6262u), c23 = prmt(z2, z3, 0x6262u);
      L.r[w][p][0] = prmt(a01, a23, 0x5410u);
      L.r[w][p][1] = prmt(a01, a23, 0x7632u);
      L.r[w][p][2] = prmt(c01, c23, 0x5410u);
    }
#pragma unroll
  for (int l = 0; l < 3; l++) {
    int se = 0, so = 0;
#pragma unroll
    for (int w = 0; w < 2; w++) {
      se = dp4a_ss(L.r[w][0][l], 0x01010101u, se);
      so = dp4a_ss(L.r[w][1][l], 0x01010101u, so);
    }
    L.a0[l] = -8 * se;
    L.b0[l] = -128 * so;
  }
  L.k01 = (finite && M > 0.f) ? __int_as_float((127 - q - 4) << 23) : 0.f;
  L.k2 = (finite && M > 0.f) ? __int_as_float((127 + 12 - q) << 23) : 0.f;
  return finite;
}

// Bounded wait that records COLI_E_TIMEOUT and sets `stop` when it gives up (a stopped role waits
// no more and its results are discarded: the call reports the error).
__device__ __forceinline__ void role_wait(uint64_t* bar, uint32_t parity, uint64_t lim, bool& stop, int* err) {
  if (!stop && !mbar_wait_suspend(bar, parity, lim)) {
    stop = true;
    set_error(err, COLI_E_TIMEOUT);
  }
}

template <int MAXT>
__global__ void __launch_bounds__(MAXT, 1) stream_ffn_kernel(const StreamParams P) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  StreamCtrl& cs = *reinterpret_cast<StreamCtrl*>(base);
  uint8_t* ring_g = base + (sizeof(StreamCtrl) + 127) / 128 * 128;
  uint8_t* ring_d = ring_g + (size_t)P.nsg * P.sbg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = P.D, NW = D / 512, NCT = 32 * NW;  // warps and threads of a consumer role
  const int C = D / 32;                            // activation chunks = 16 NW
  const uint32_t pitch = (uint32_t)D / 2;          // bytes of a gate/up row
  const uint32_t rows_bytes = 16u * pitch;         // a unit's 16 gate (or up) rows = its down panel
  const int NSG = P.nsg, NSD = P.nsd;
  const uint64_t lim = P.wait_ns ? P.wait_ns : kWaitLimitNs;
  const int W_PG = 2 * NW, W_PD = 2 * NW + 1, W_H = 2 * NW + 2;  // producer warps and the h warp

  if (tid == 0) {
    for (int s = 0; s < NSG; s++) {
      mbar_init(&cs.full_g[s], 1);
      mbar_init(&cs.empty_g[s], NW);
    }
    for (int s = 0; s < NSD; s++) {
      mbar_init(&cs.full_d[s], 1);
      mbar_init(&cs.empty_d[s], NW);
    }
    for (int b = 0; b < kHB; b++) {
      mbar_init(&cs.redf[b], NCT);
      mbar_init(&cs.redfree[b], 1);
      mbar_init(&cs.hlf[b], 1);
      mbar_init(&cs.hlfree[b], NW);
    }
    mbar_init(&cs.xfull, 1);
    mbar_init(&cs.xfree, NW);
    mbar_fence_init();
    // x (the router's input, complete before this grid started) into gate/up stage 0 with one bulk
    // copy: every CTA needs all of it, and 152 CTAs of per-thread loads of the same 24 KiB queue for
    // microseconds behind each other in L2, where one bulk request per CTA does not
    if (P.x_bulk) {
      const uint32_t xbytes = (uint32_t)D * (P.x_dtype == COLI_DTYPE_F32 ? 4u : 2u);
      mbar_arrive_expect_tx(&cs.xfull, xbytes);
      bulk_g2s(ring_g, P.x, xbytes, &cs.xfull);
    }
  }
  __syncthreads();  // the barriers are initialised before any thread waits on or arrives at one
  // gate/up prologue, overlapping the router's tail: the limbs of this thread's chunk of x
  const int c = tid % C, r0 = tid / C;  // gate/up threads: r0 in {0, 1}
  Limbs X;
  if (warp < NW) {
    float xv[32];
    if (P.x_bulk) {
      __syncwarp();
      bool late = false;
      role_wait(&cs.xfull, 0, lim, late, P.err);
      if (P.x_dtype == COLI_DTYPE_F32) {  // chunk c: 32 floats at byte 128 c
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const uint4 u = lds128(ring_g + 128 * c + 16 * i);
          xv[4 * i] = __uint_as_float(u.x);
          xv[4 * i + 1] = __uint_as_float(u.y);
          xv[4 * i + 2] = __uint_as_float(u.z);
          xv[4 * i + 3] = __uint_as_float(u.w);
        }
      } else {  // 32 bf16 at byte 64 c
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const uint4 u = lds128(ring_g + 64 * c + 16 * i);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int h = 0; h < 4; h++) {
            xv[8 * i + 2 * h] = __uint_as_float(w4[h] << 16);
            xv[8 * i + 2 * h + 1] = __uint_as_float(w4[h] & 0xffff0000u);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cs.xfree);  // stage 0 may be refilled
    } else {
      load_chunk_f32(P.x, P.x_dtype, 0, 32 * c, D, xv);
    }
    if (!make_limbs(xv, X)) set_error(P.err, COLI_E_NONFINITE);
  }
  griddep_wait();  // idx, w and n_sel come from the router
  // Slots from the routes in two rounds of loads: the kept count, the expert ids and the weights
  // together, then every table field a slot needs, read whether or not the entry turns out valid
  // (the id is clamped into the table), so that no load waits for another's answer.
  if (tid < P.K) {
    const int m_raw = P.n_sel ? ld_cg_i32(P.n_sel) : P.K;
    const int e = ld_cg_i32(P.idx + tid);
    const float wk = ld_cg_f32(P.w + tid);
    const int m = m_raw < 0 ? 0 : (m_raw > P.K ? P.K : m_raw);
    if (tid == 0) cs.m = m;
    if (tid < m) {
      const bool in_table = e >= 0 && e < COLI_MAX_EXPERTS;
      const ExpertDesc* ed = P.table + (in_table ? e : 0);
      const TensorDesc* g = &ed->t[T_GATE];
      const TensorDesc* u = &ed->t[T_UP];
      const TensorDesc* d = &ed->t[T_DOWN];
      // every field into registers first (read-only loads, none ordered after a shared-memory store)
      const int valid = __ldg(&ed->valid);
      const uint8_t* gw = reinterpret_cast<const uint8_t*>(__ldg(reinterpret_cast<const unsigned long long*>(&g->w)));
      const uint8_t* uw = reinterpret_cast<const uint8_t*>(__ldg(reinterpret_cast<const unsigned long long*>(&u->w)));
      const uint8_t* dp = reinterpret_cast<const uint8_t*>(__ldg(reinterpret_cast<const unsigned long long*>(&d->panel)));
      const float* gsc = reinterpret_cast<const float*>(__ldg(reinterpret_cast<const unsigned long long*>(&g->s)));
      const float* usc = reinterpret_cast<const float*>(__ldg(reinterpret_cast<const unsigned long long*>(&u->s)));
      const float* dsr = reinterpret_cast<const float*>(__ldg(reinterpret_cast<const unsigned long long*>(&d->s)));
      const float* dst = reinterpret_cast<const float*>(__ldg(reinterpret_cast<const unsigned long long*>(&d->sT)));
      const int gmode = __ldg(&g->mode), umode = __ldg(&u->mode), dmode = __ldg(&d->mode);
      const int Gg = __ldg(&g->G), Gu = __ldg(&u->G);
      const int gsg = __ldg(&g->gs), gsu = __ldg(&u->gs), gsd = __ldg(&d->gs);
      StreamSlot& sl = cs.slot[tid];
      sl.gw = gw;
      sl.uw = uw;
      sl.dp = dp;
      sl.gs = gsc;
      sl.us = usc;
      sl.gmode = gmode;
      sl.umode = umode;
      sl.dmode = dmode;
      sl.ds = dmode == SCALE_ROW ? dsr : dst;
      sl.Gg = Gg;
      sl.Gu = Gu;
      sl.gsg = gsg;
      sl.gsu = gsu;
      sl.gsd = gsd;
      sl.wk = wk;
      bool ok = in_table && valid;
      if (!ok) set_error(P.err, COLI_E_ROUTE);
      // the host launches this kernel only for tables it can stream; anything else is a bad entry
      if (ok && (gmode == SCALE_GENERIC || umode == SCALE_GENERIC || dmode == SCALE_GENERIC || !dp ||
                 !(dmode == SCALE_ROW ? dsr : dst) || rows_bytes + 64u * Gg > P.sbg || rows_bytes + 64u * Gu > P.sbg)) {
        ok = false;
        set_error(P.err, COLI_E_ROUTE);
      }
      sl.ok = ok;
    }
  }
  __syncthreads();
  griddep_launch_dependents();  // the reduce kernel may launch; it waits for this grid to finish
  const int m = cs.m;

  const int UB = P.I / kPanelCols;  // units per slot
  const long long total = (long long)m * UB;
  const int ubeg = (int)((long long)blockIdx.x * total / gridDim.x);
  const int uend = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
  bool stop = false;

  if (warp == W_PG || warp == W_PD) {
    // ---------------- producers: one lane per ring issues its copies in unit order ----------------
    if (lane == 0) {
      const bool gu = warp == W_PG;
      const uint64_t pol = l2_evict_first_policy();
      uint64_t* full = gu ? cs.full_g : cs.full_d;
      uint64_t* empty = gu ? cs.empty_g : cs.empty_d;
      uint8_t* ring = gu ? ring_g : ring_d;
      const int NS = gu ? NSG : NSD;
      const uint32_t SB = gu ? P.sbg : P.sbd;
      uint32_t q = 0, s = 0, ph = 0;  // stage sequence number, its slot and the slot's use parity
      bool withhold = gu && P.withhold && ubeg == 0 && uend > 0;  // the CTA that owns unit 0
      if (gu && P.x_bulk) role_wait(&cs.xfree, 0, lim, stop, P.err);  // x has left stage 0
      // one stage of up to two pieces (weights, then their scales) on one barrier
      auto issue = [&](const void* src, uint32_t bytes, const void* src2, uint32_t bytes2, bool weights) {
        if (stop) return;
        if (q >= (uint32_t)NS) role_wait(&empty[s], ph ^ 1u, lim, stop, P.err);
        if (stop) return;
        mbar_arrive_expect_tx(&full[s], bytes + bytes2);
        uint8_t* dst = ring + (size_t)s * SB;
        if (withhold) {  // test hook: the stage never fills, so its consumers' bounded waits give up
          withhold = false;
        } else {
          if (weights)
            bulk_g2s_stream(dst, src, bytes, &full[s], pol);
          else
            bulk_g2s(dst, src, bytes, &full[s]);
          if (bytes2) bulk_g2s(dst + bytes, src2, bytes2, &full[s]);
        }
        q++;
        if (++s == (uint32_t)NS) {
          s = 0;
          ph ^= 1u;
        }
      };
      int prev = -1;
      for (int u = ubeg; u < uend && !stop; u++) {
        const int j = u / UB, b = u - j * UB;
        const StreamSlot& sl = cs.slot[j];
        if (!sl.ok) continue;
        const int i0 = b * kPanelCols;
        if (gu) {  // the rows, then their 16 row scales or 16 rows of chunk-group scales
          issue(sl.gw + (size_t)i0 * pitch, rows_bytes, sl.gs + (size_t)i0 * sl.Gg, 64u * sl.Gg, true);
          issue(sl.uw + (size_t)i0 * pitch, rows_bytes, sl.us + (size_t)i0 * sl.Gu, 64u * sl.Gu, true);
        } else {
          if (sl.dmode == SCALE_CHUNK || j != prev)  // down scales when they change
            issue(sl.dmode == SCALE_CHUNK ? sl.ds + (size_t)(i0 / sl.gsd) * D : sl.ds, 4u * D, nullptr, 0u, false);
          issue(sl.dp + (size_t)b * rows_bytes, rows_bytes, nullptr, 0u, true);
        }
        prev = j;
      }
      // never leave with copies in flight into the ring (a withheld stage is given up on, bounded)
      for (uint32_t r = q > (uint32_t)NS ? q - NS : 0; r < q; r++)
        (void)mbar_wait_suspend(&full[r % NS], (r / NS) & 1, lim);
    }
  } else if (warp == W_H) {
    // ---------------- h warp: row sums -> h = SiLU(g s_g) (u s_u) -> limbs ----------------
    int n = 0;
    for (int u = ubeg; u < uend; u++) {
      if (!cs.slot[u / UB].ok) continue;
      const int b = n % kHB;
      const uint32_t use = (uint32_t)(n / kHB);
      role_wait(&cs.redf[b], use & 1, lim, stop, P.err);
      float h = 0.f;
      if (lane < 16) {
        // row `lane` = r0 + 2 i of the unit is value i (gate) and 8 + i (up) of the warps with that r0
        const int rg = lane & 1, v = lane >> 1;
        float g = 0.f, uu = 0.f;
        for (int w = rg * (NW / 2); w < (rg + 1) * (NW / 2); w++) {
          g += cs.red[b][w][v];
          uu += cs.red[b][w][8 + v];
        }
        h = silu_mul(g * cs.fs[b][0][lane], uu * cs.fs[b][1][lane]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cs.redfree[b]);  // the gate/up warps may refill buffer b
      Limbs16 L;
      const bool fin = warp_limbs16(h, lane, L);
      if (use >= 1) role_wait(&cs.hlfree[b], (use - 1) & 1, lim, stop, P.err);
      if (lane == 0) {
        if (!fin && !stop) set_error(P.err, COLI_E_NONFINITE);
        cs.hl[b] = L;
        mbar_arrive(&cs.hlf[b]);
      }
      n++;
    }
  } else if (warp < NW) {
    // ---------------- gate/up warps ----------------
    uint32_t s = 0, ph = 0;  // ring slot of the next stage and its use parity
    int n = 0;
    for (int u = ubeg; u < uend; u++) {
      const StreamSlot& sl = cs.slot[u / UB];
      if (!sl.ok) continue;
      const int b = n % kHB;
      const uint32_t use = (uint32_t)(n / kHB);
      // gate, then up: rows r0 + 2 i (i < 8) of the unit, this thread's chunk; the stage's 16 rows are
      // followed by their scales (one per row, or one per chunk group and row). Each stage's eight values
      // are summed over the warp at once: lanes 4 i .. 4 i + 3 end with value i, gate (or up) row r0 + 2 i.
#pragma unroll
      for (int t = 0; t < 2; t++) {
        role_wait(&cs.full_g[s], ph, lim, stop, P.err);
        const uint8_t* st = ring_g + (size_t)s * P.sbg;
        const float* sc = reinterpret_cast<const float*>(st + rows_bytes);
        const int mode = t ? sl.umode : sl.gmode, G = t ? sl.Gu : sl.Gg;
        const int grp = mode == SCALE_CHUNK ? (32 * c) / (t ? sl.gsu : sl.gsg) : 0;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
          float d = chunk_dot(lds128(st + (r0 + 2 * i) * pitch + 16 * c), X);
          if (mode == SCALE_CHUNK) d *= sc[(r0 + 2 * i) * G + grp];
          v[i] = d;
        }
        if (t == 0 && use >= 1) role_wait(&cs.redfree[b], (use - 1) & 1, lim, stop, P.err);  // buffer b is free
        if (warp == 0 && lane < 16) cs.fs[b][t][lane] = mode == SCALE_ROW ? sc[lane] : 1.f;
        __syncwarp();
        if (lane == 0 && !stop) mbar_arrive(&cs.empty_g[s]);
        if (++s == (uint32_t)NSG) {
          s = 0;
          ph ^= 1u;
        }
        warp_transpose_reduce<8>(v, lane);
        if (!(lane & 3)) cs.red[b][warp][8 * t + (lane >> 2)] = v[0];
      }
      mbar_arrive(&cs.redf[b]);
      n++;
    }
  } else if (warp < 2 * NW) {
    // ---------------- down warps ----------------
    const int td = tid - NCT;  // rows td + jj NCT of y
    float acc[16], ws[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      acc[i] = 0.f;
      ws[i] = 0.f;
    }
    uint32_t s = 0, ph = 0;
    auto next_stage = [&]() {
      if (++s == (uint32_t)NSD) {
        s = 0;
        ph ^= 1u;
      }
    };
    int n = 0, prev = -1;
    for (int u = ubeg; u < uend; u++) {
      const int j = u / UB;
      const StreamSlot& sl = cs.slot[j];
      if (!sl.ok) continue;
      const int b = n % kHB;
      const uint32_t use = (uint32_t)(n / kHB);
      if (sl.dmode == SCALE_CHUNK || j != prev) {  // w_k times the down scales of this thread's rows
        role_wait(&cs.full_d[s], ph, lim, stop, P.err);
        const float* sd = reinterpret_cast<const float*>(ring_d + (size_t)s * P.sbd);
#pragma unroll
        for (int jj = 0; jj < 16; jj++) ws[jj] = sl.wk * sd[td + jj * NCT];
        __syncwarp();
        if (lane == 0 && !stop) mbar_arrive(&cs.empty_d[s]);
        next_stage();
      }
      prev = j;
      role_wait(&cs.hlf[b], use & 1, lim, stop, P.err);
      const Limbs16 HL = cs.hl[b];
      __syncwarp();
      if (lane == 0) mbar_arrive(&cs.hlfree[b]);
      role_wait(&cs.full_d[s], ph, lim, stop, P.err);
      const uint8_t* st = ring_d + (size_t)s * P.sbd;
#pragma unroll
      for (int jj = 0; jj < 16; jj++) {
        const uint2 wv = lds64(st + (size_t)(td + jj * NCT) * 8);
        acc[jj] = fmaf(ws[jj], chunk_dot16(wv, HL), acc[jj]);
      }
      __syncwarp();
      if (lane == 0 && !stop) mbar_arrive(&cs.empty_d[s]);
      next_stage();
      n++;
    }
    float* prow = P.part + (size_t)blockIdx.x * D;
#pragma unroll
    for (int jj = 0; jj < 16; jj++) prow[td + jj * NCT] = acc[jj];
  }
}

// y[d] = resid[d] + (sum over the G partial rows of column d, in CTA order). A CTA takes 32 columns;
// its eight warps add eight consecutive runs of the partial rows, then the runs are added in order.
__global__ void __launch_bounds__(256) stream_reduce_kernel(const float* __restrict__ part, int G, int D,
                                                            const void* resid, int x_dtype, void* y, int y_dtype) {
  __shared__ float fold[8][32];
  griddep_wait();  // every partial row is stored
  const int dl = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int d = blockIdx.x * 32 + dl;
  float s = 0.f;
  if (d < D) {
    const int c0 = grp * G / 8, c1 = (grp + 1) * G / 8;
#pragma unroll 8
    for (int cc = c0; cc < c1; cc++) s += __ldcg(part + (size_t)cc * D + d);
  }
  fold[grp][dl] = s;
  __syncthreads();
  if (grp == 0 && d < D) {
    float tot = fold[0][dl];
#pragma unroll
    for (int g2 = 1; g2 < 8; g2++) tot += fold[g2][dl];
    if (resid) tot = load_act(resid, x_dtype, d) + tot;
    if (y_dtype == COLI_DTYPE_F32)
      static_cast<float*>(y)[d] = tot;
    else
      static_cast<uint16_t*>(y)[d] = f32_to_bf16_rn(tot);
  }
}

// ------------------------------------------------------------------------------------------
// One token through a dense int4 tensor, y = resid + W x (coli_w4_linear with S = 1): the gate/up role
// of the streaming FFN on its own. Units of 16 rows; CTA c streams the rows of its contiguous range of
// units through a ring of bulk-copied stages (16 rows and their scales each); NW row warps dot them with
// x's limbs (one 32-column chunk per thread, rows r0 + 2i, i < 8) and leave each warp's row sums; a
// finishing warp adds a row's warp sums in warp order, applies the row scale and the residual and writes
// y. A unit's rows belong to one CTA, so no CTA waits for another and no reduce follows.
// ------------------------------------------------------------------------------------------

constexpr int kLinStages = 3;

struct LinCtrl {
  uint64_t full[kLinStages], empty[kLinStages];
  uint64_t redf[kHB], redfree[kHB];
  uint64_t xfull;
  float red[kHB][kStMaxWarps][8];  // per row warp: its 8 row sums of a unit
  float fs[kHB][16];
};

struct LinParams {
  const uint8_t* w;  // rows of I/2 bytes
  const float* s;    // per-row scales, or G per row
  const void* x;
  const void* resid;
  void* y;
  int* err;
  int O, I, G, gs, mode, x_dtype, x_bulk;
  uint32_t sb;       // stage bytes
  unsigned long long wait_ns;
};

__global__ void __launch_bounds__(448, 1) stream_linear_kernel(const LinParams P) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  LinCtrl& cs = *reinterpret_cast<LinCtrl*>(base);
  uint8_t* xbuf = base + (sizeof(LinCtrl) + 127) / 128 * 128;
  uint8_t* ring = xbuf + (size_t)P.I * 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int I = P.I, NW = I / 512, NCT = 32 * NW, C = I / 32;
  const uint32_t pitch = (uint32_t)I / 2, rows_bytes = 16u * pitch;
  const uint64_t lim = P.wait_ns ? P.wait_ns : kWaitLimitNs;
  const int W_P = NW, W_F = NW + 1;  // producer warp, finishing warp
  if (tid == 0) {
    for (int s = 0; s < kLinStages; s++) {
      mbar_init(&cs.full[s], 1);
      mbar_init(&cs.empty[s], NW);
    }
    for (int b = 0; b < kHB; b++) {
      mbar_init(&cs.redf[b], NCT);
      mbar_init(&cs.redfree[b], 1);
    }
    mbar_init(&cs.xfull, 1);
    mbar_fence_init();
    if (P.x_bulk) {
      const uint32_t xbytes = (uint32_t)I * (P.x_dtype == COLI_DTYPE_F32 ? 4u : 2u);
      mbar_arrive_expect_tx(&cs.xfull, xbytes);
      bulk_g2s(xbuf, P.x, xbytes, &cs.xfull);
    }
  }
  __syncthreads();
  const int U = P.O / 16;
  const int ubeg = (int)((long long)blockIdx.x * U / gridDim.x), uend = (int)((long long)(blockIdx.x + 1) * U / gridDim.x);
  bool stop = false;
  if (warp < NW) {
    // ---------------- row warps ----------------
    const int c = tid % C, r0 = tid / C;
    Limbs X;
    {
      float xv[32];
      if (P.x_bulk) {
        bool late = false;
        role_wait(&cs.xfull, 0, lim, late, P.err);
        if (P.x_dtype == COLI_DTYPE_F32) {
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const uint4 u = lds128(xbuf + 128 * c + 16 * i);
            xv[4 * i] = __uint_as_float(u.x);
            xv[4 * i + 1] = __uint_as_float(u.y);
            xv[4 * i + 2] = __uint_as_float(u.z);
            xv[4 * i + 3] = __uint_as_float(u.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const uint4 u = lds128(xbuf + 64 * c + 16 * i);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int h = 0; h < 4; h++) {
              xv[8 * i + 2 * h] = __uint_as_float(w4[h] << 16);
              xv[8 * i + 2 * h + 1] = __uint_as_float(w4[h] & 0xffff0000u);
            }
          }
        }
      } else {
        load_chunk_f32(P.x, P.x_dtype, 0, 32 * c, I, xv);
      }
      if (!make_limbs(xv, X)) set_error(P.err, COLI_E_NONFINITE);
    }
    const int grp = P.mode == SCALE_CHUNK ? (32 * c) / P.gs : 0;
    uint32_t s = 0, ph = 0;
    int n = 0;
    for (int u = ubeg; u < uend && !stop; u++) {
      const int b = n % kHB;
      const uint32_t use = (uint32_t)(n / kHB);
      role_wait(&cs.full[s], ph, lim, stop, P.err);
      const uint8_t* st = ring + (size_t)s * P.sb;
      const float* sc = reinterpret_cast<const float*>(st + rows_bytes);
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        float d = chunk_dot(lds128(st + (r0 + 2 * i) * pitch + 16 * c), X);
        if (P.mode == SCALE_CHUNK) d *= sc[(r0 + 2 * i) * P.G + grp];
        v[i] = d;
      }
      if (use >= 1) role_wait(&cs.redfree[b], (use - 1) & 1, lim, stop, P.err);
      if (warp == 0 && lane < 16) cs.fs[b][lane] = P.mode == SCALE_ROW ? sc[lane] : 1.f;
      __syncwarp();
      if (lane == 0 && !stop) mbar_arrive(&cs.empty[s]);
      if (++s == (uint32_t)kLinStages) {
        s = 0;
        ph ^= 1u;
      }
      warp_transpose_reduce<8>(v, lane);
      if (!(lane & 3)) cs.red[b][warp][lane >> 2] = v[0];
      mbar_arrive(&cs.redf[b]);
      n++;
    }
  } else if (warp == W_P) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t sbytes = P.mode == SCALE_ROW ? 64u : 64u * (uint32_t)P.G;
      uint32_t q = 0, s = 0, ph = 0;
      for (int u = ubeg; u < uend && !stop; u++) {
        if (q >= (uint32_t)kLinStages) role_wait(&cs.empty[s], ph ^ 1u, lim, stop, P.err);
        if (stop) break;
        mbar_arrive_expect_tx(&cs.full[s], rows_bytes + sbytes);
        uint8_t* dst = ring + (size_t)s * P.sb;
        bulk_g2s_stream(dst, P.w + (size_t)u * rows_bytes, rows_bytes, &cs.full[s], pol);
        bulk_g2s(dst + rows_bytes, P.s + (size_t)u * 16 * (P.mode == SCALE_ROW ? 1 : P.G), sbytes, &cs.full[s]);
        q++;
        if (++s == (uint32_t)kLinStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      for (uint32_t r = q > (uint32_t)kLinStages ? q - kLinStages : 0; r < q; r++)
        (void)mbar_wait_suspend(&cs.full[r % kLinStages], (r / kLinStages) & 1, lim);
    }
  } else if (warp == W_F) {
    // ---------------- finishing warp: row sums -> y ----------------
    int n = 0;
    for (int u = ubeg; u < uend && !stop; u++) {
      const int b = n % kHB;
      role_wait(&cs.redf[b], (uint32_t)(n / kHB) & 1, lim, stop, P.err);
      if (lane < 16 && !stop) {
        // row `lane` = r0 + 2 i of the unit is value i of the warps with that r0
        const int rg = lane & 1, v = lane >> 1;
        float t = 0.f;
        for (int w = rg * (NW / 2); w < (rg + 1) * (NW / 2); w++) t += cs.red[b][w][v];
        t *= cs.fs[b][lane];
        const int row = 16 * u + lane;
        if (P.resid) t = load_act(P.resid, P.x_dtype, row) + t;
        if (P.x_dtype == COLI_DTYPE_F32)
          static_cast<float*>(P.y)[row] = t;
        else
          static_cast<uint16_t*>(P.y)[row] = f32_to_bf16_rn(t);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cs.redfree[b]);
      n++;
    }
  }
  // never leave with the x copy in flight (it completes before any row warp starts; bounded)
  if (tid == 0 && P.x_bulk) (void)mbar_wait_suspend(&cs.xfull, 0, lim);
}

bool stream_linear_ok(const HostTensor& t) {
  return t.I % 1024 == 0 && t.I <= 512 * kStMaxWarps && t.O % 16 == 0 && (t.gs == 0 || t.gs % 32 == 0) &&
         t.pitch == (uint32_t)t.I / 2;
}

int launch_stream_linear(coli_ctx* ctx, const HostTensor& t, const void* x, int x_dtype, const void* resid, void* y) {
  LinParams P;
  P.w = t.w;
  P.s = t.s;
  P.x = x;
  P.resid = resid;
  P.y = y;
  P.err = ctx->d_status;
  P.O = t.O;
  P.I = t.I;
  P.G = t.G;
  P.gs = t.gs;
  P.mode = t.desc.mode;
  P.x_dtype = x_dtype;
  P.x_bulk = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  P.sb = (uint32_t)align_up(16u * (uint32_t)t.I / 2 + 64u * (uint32_t)t.G, 128);
  P.wait_ns = ctx->wait_ns;
  const int NW = t.I / 512;
  const size_t smem = 128 + align_up(sizeof(LinCtrl), 128) + (size_t)t.I * 4 + (size_t)kLinStages * P.sb;
  cudaError_t e = cudaFuncSetAttribute(stream_linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream linear: shared memory attribute");
  int grid = ctx->num_sms;
  if (grid > t.O / 16) grid = t.O / 16;
  ProfScope prof(ctx, COLI_KERNEL_LINEAR);
  e = launch_k(stream_linear_kernel, grid, 32 * (NW + 2), smem, ctx->stream, false, false, P);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream linear launch");
  return COLI_OK;
}

// ------------------------------------------------------------------------------------------
// Panel-major view of a down tensor: column block p (kPanelCols columns) of every row, contiguous.
// ------------------------------------------------------------------------------------------

__global__ void panel_kernel(const uint8_t* __restrict__ w, uint32_t pitch, int rows, int npanels,
                             uint8_t* __restrict__ panel) {
  const long long n = (long long)npanels * rows;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(i / rows), d = (int)(i - (long long)p * rows);
    const uint2 v = *reinterpret_cast<const uint2*>(w + (size_t)d * pitch + (size_t)p * (kPanelCols / 2));
    *reinterpret_cast<uint2*>(panel + (size_t)i * (kPanelCols / 2)) = v;
  }
}

__global__ void transpose_scales_kernel(const float* __restrict__ s, int rows, int G, float* __restrict__ sT) {
  const long long n = (long long)rows * G;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(i / rows), d = (int)(i - (long long)g * rows);
    sT[i] = s[(size_t)d * G + g];
  }
}

static constexpr size_t stream_ctrl_bytes() { return (sizeof(StreamCtrl) + 127) / 128 * 128; }

bool stream_tensor_ok(const HostTensor& t, bool as_down) {
  if (!(t.gs == 0 || t.gs % 32 == 0)) return false;
  if (as_down) return t.O % 1024 == 0 && t.O <= 512 * kStMaxWarps && t.I % kPanelCols == 0;  // [D x I]
  return t.I % 1024 == 0 && t.I <= 512 * kStMaxWarps && t.O % kPanelCols == 0;              // [I x D]
}

int build_stream_view(coli_ctx* ctx, HostTensor& t) {
  if (t.panel) return COLI_OK;
  const int npanels = t.I / kPanelCols;
  const size_t pbytes = (size_t)npanels * t.O * (kPanelCols / 2);
  void* pp = nullptr;
  void* ps = nullptr;
  cudaError_t e = cudaMalloc(&pp, pbytes);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "table_set: cudaMalloc down panels");
  if (t.gs > 0 && (e = cudaMalloc(&ps, (size_t)t.O * t.G * sizeof(float))) != cudaSuccess) {
    cudaFree(pp);
    return cuda_fail(ctx, e, "table_set: cudaMalloc transposed scales");
  }
  const long long n = (long long)npanels * t.O;
  int grid = (int)((n + 255) / 256);
  if (grid > 8 * ctx->num_sms) grid = 8 * ctx->num_sms;
  panel_kernel<<<grid, 256, 0, ctx->stream>>>(t.w, t.pitch, t.O, npanels, static_cast<uint8_t*>(pp));
  if (ps) {
    const long long ns = (long long)t.O * t.G;
    int g2 = (int)((ns + 255) / 256);
    if (g2 > 8 * ctx->num_sms) g2 = 8 * ctx->num_sms;
    transpose_scales_kernel<<<g2, 256, 0, ctx->stream>>>(t.s, t.O, t.G, static_cast<float*>(ps));
  }
  if ((e = cudaGetLastError()) != cudaSuccess || (e = cudaStreamSynchronize(ctx->stream)) != cudaSuccess) {
    cudaFree(pp);
    if (ps) cudaFree(ps);
    return cuda_fail(ctx, e, "table_set: build down panels");
  }
  t.panel = static_cast<uint8_t*>(pp);
  t.sT = static_cast<float*>(ps);
  t.desc.panel = t.panel;
  t.desc.sT = t.sT;
  return COLI_OK;
}

// Ring sizes: a gate/up stage holds a unit's 16 rows and their scales, a down stage a unit's panel
// (or its down scales); both rings get the same number of stages, as many as fit.
static bool stream_rings(const coli_ctx* ctx, int D, uint32_t& sbg, uint32_t& sbd, int& ns, size_t& smem) {
  int maxsm = 0;
  if (cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  const int gmax = ctx->table_gu_maxG > 1 ? ctx->table_gu_maxG : 1;
  sbg = (uint32_t)align_up(8u * (uint32_t)D + 64u * (uint32_t)gmax, 128);
  sbd = 8u * (uint32_t)D;
  const long long room = (long long)maxsm - 128 - (long long)stream_ctrl_bytes();
  ns = (int)(room / ((long long)sbg + sbd));
  if (ns > kStMaxStages) ns = kStMaxStages;
  smem = 128 + stream_ctrl_bytes() + (size_t)ns * (sbg + sbd);
  return ns >= 2;
}

bool stream_eligible(const coli_ctx* ctx, int S) {
  const int D = ctx->table_D, I = ctx->table_I;
  uint32_t sbg, sbd;
  int ns;
  size_t smem;
  return S == 1 && ctx->stream_ffn && !ctx->decode_fused && ctx->table_count > 0 && ctx->table_nostream == 0 &&
         D % 1024 == 0 && D <= 512 * kStMaxWarps && I % kPanelCols == 0 && stream_rings(ctx, D, sbg, sbd, ns, smem);
}

int launch_stream_ffn(coli_ctx* ctx, const void* x, int x_dtype, const int32_t* idx, const float* w,
                      const int32_t* n_sel, int K, const void* resid, void* y, int y_dtype) {
  const int D = ctx->table_D, I = ctx->table_I;
  const int NW = D / 512, threads = 32 * (2 * NW + 3);
  uint32_t sbg, sbd;
  int ns;
  size_t smem;
  if (!stream_rings(ctx, D, sbg, sbd, ns, smem)) return fail(ctx, COLI_E_INVAL, "stream FFN: rings do not fit");
  auto kern = threads <= 480 ? stream_ffn_kernel<480> : stream_ffn_kernel<864>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return cuda_fail(ctx, e, "stream FFN: shared memory attribute");
  const int G = ctx->num_sms;
  int rc = ensure_workspace(ctx, (size_t)G * D * sizeof(float));
  if (rc != COLI_OK) return rc;
  StreamParams P;
  P.x = x;
  P.x_dtype = x_dtype;
  P.D = D;
  P.I = I;
  P.K = K;
  P.idx = idx;
  P.w = w;
  P.n_sel = n_sel;
  P.table = ctx->d_table;
  P.part = reinterpret_cast<float*>(ctx->ws.base);
  P.err = ctx->d_status;
  P.nsg = P.nsd = ns;
  P.sbg = sbg;
  P.sbd = sbd;
  P.wait_ns = ctx->wait_ns;
  P.withhold = ctx->test_withhold > 0;  // one-shot: only the next launch withholds
  P.x_bulk = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  if (ctx->test_withhold > 0) ctx->test_withhold--;
  {
    ProfScope prof(ctx, COLI_KERNEL_GATEUP);
    e = launch_k(kern, G, threads, smem, ctx->stream, true, false, P);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream FFN launch");
  {
    ProfScope prof(ctx, COLI_KERNEL_COMBINE);
    e = launch_k(stream_reduce_kernel, (D + 31) / 32, 256, 0, ctx->stream, true, false,
                 static_cast<const float*>(P.part), G, D, resid, x_dtype, y, y_dtype);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream FFN reduce launch");
  return COLI_OK;
}

}  // namespace coli
