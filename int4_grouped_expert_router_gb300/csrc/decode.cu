// S = 1 decode: the whole grouped int4 expert FFN of one token -- gate + up dual GEMV, SiLU(g) * u,
// the down GEMV, per-expert weighting and a fixed-order reduce into the residual -- in one
// persistent launch that streams every kept expert's weights once.
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
// another CTA's h, so each CTA's weight stream runs from its first unit to its last without a
// dependency bubble. At the end every CTA stores its partial row, the grid meets once (a cooperative
// launch: every CTA is resident) and CTA c adds the partial rows of its share of y in CTA order,
// then the residual: a fixed-order, atomics-free reduce, bit-identical from run to run.
//
// Streaming. One producer lane per CTA copies the unit's blocks into a ring of shared-memory stages
// with bulk asynchronous copies (cp.async.bulk, completion on an mbarrier); every stage is 2 D
// bytes: four gate or up rows (a row is D / 2 bytes), or a quarter of the down panel (D / 4 rows of
// 8 bytes), or scales. The consumer warps (D / 512 of them, one activation chunk of 32 columns per
// thread, two thread rows) never leave the ring: each stage is released to the producer as soon as
// every warp has read it, and every wait suspends the warp in mbarrier.try_wait rather than polling.
// A separate warp turns each unit's row sums into h while the consumers stream the next unit.
//
// Arithmetic: the block-fixed-point dp4a dot product of dot.h. Gate and up use 32-column chunks of
// x; the down projection uses the unit's 16 values of h as one 16-column block (its own power-of-two
// scale), so each down dot product has the same error bound as a chunk of the gate/up ones.
#include "coli_internal.h"
#include "dot.h"
#include "pipe.h"

namespace coli {

constexpr int kStMaxStages = 32;
constexpr int kStMinStages = 3;   // one stage read, two in flight
constexpr int kStMaxWarps = 16;   // consumer warps: D <= 8192
constexpr int kLag = 2;           // a unit's down stage follows the gate/up stages of the unit kLag later

struct StreamSlot {
  const uint8_t* gw;  // gate rows [I x D/2]
  const uint8_t* uw;  // up rows [I x D/2]
  const uint8_t* dp;  // down panels [I/16][D][8 bytes]
  const float* gs;    // gate scales: [I] (per row) or [I x Gg] (chunk groups)
  const float* us;    // up scales
  const float* ds;    // down scales: [D] (per row) or transposed chunk-group scales [Gd x D]
  float wk;           // routing weight of the slot
  int gmode, umode, dmode;
  int Gg, Gu;         // groups per gate / up row
  int gsg, gsu, gsd;  // group sizes (0: per row)
  int ok;
};

struct StreamCtrl {
  uint64_t full[kStMaxStages];   // stage holds data (producer's expect_tx + the copies' bytes)
  uint64_t empty[kStMaxStages];  // every consumer warp has read the stage
  uint64_t redf[kLag + 1];       // every consumer thread has stored its row sums of unit n (buffer n % 3)
  uint64_t hlf[kLag + 1];        // the h warp has stored the limbs of that unit's h
  StreamSlot slot[COLI_MAX_K];
  float red[kLag + 1][kStMaxWarps][16];  // per consumer warp: its 8 gate and 8 up row sums of a unit
  Limbs16 hl[kLag + 1];                  // h of a unit as one 16-column block of limbs
  float fold[32 * (kStMaxWarps + 2)];  // final reduce: group sums
  int m;
};

struct StreamParams {
  const void* x;
  int x_dtype, y_dtype;
  int D, I, K;
  const int32_t* idx;
  const float* w;
  const int32_t* n_sel;
  const ExpertDesc* table;
  const void* resid;
  void* y;
  float* part;               // [gridDim.x x D] partial rows
  unsigned long long* bar;   // grid barrier count (monotonic)
  int* err;
  int nst;                   // ring stages
  uint32_t sb;               // stage bytes: 16 gate/up rows and their chunk scales, a down panel (8 D)
  unsigned long long wait_ns;
  int withhold;              // test hook: CTA 0 does not arrive at the grid barrier
};

// Warp roles: warps 0 .. NW-1 consume the ring (NW = D / 512), warp NW is the producer (one lane
// issues every copy), warp NW + 1 turns each unit's row sums into h and its limbs.
//
// Order of a CTA's stream, for its kept units n = 0, 1, ... (unit n: slot j, rows i0 .. i0 + 15),
// one stage each:
//   gate rows i0 .. i0 + 15 (+ their chunk-group scales), up rows (+ scales), then for unit n - 2 its
//   down scales when they change (a new slot, or chunk-group scales) and its down panel;
// and finally the down scales and panels of the last two units. A unit's down stage thus follows the
// gate/up stages of the next two units: while the consumers stream those, the h warp turns its row
// sums into h, and no consumer waits for another. Stages are large (a whole unit's gate rows, 8 D
// bytes) so that each wait and release is paid for by eight independent chunk dot products per
// thread.
template <int MAXT>
__global__ void __launch_bounds__(MAXT, 1) stream_ffn_kernel(const StreamParams P) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 127) & ~uintptr_t(127));
  StreamCtrl& cs = *reinterpret_cast<StreamCtrl*>(base);
  uint8_t* ring = base + (sizeof(StreamCtrl) + 127) / 128 * 128;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = P.D, NW = D / 512, NCT = 32 * NW;  // consumer warps and threads
  const int C = D / 32;                            // activation chunks = 16 NW
  const uint32_t SB = P.sb;                        // stage bytes
  const uint32_t pitch = (uint32_t)D / 2;          // bytes of a gate/up row
  const uint32_t rows_bytes = 16u * pitch;         // a unit's 16 gate (or up) rows = its down panel
  const int NST = P.nst;
  const uint64_t lim = P.wait_ns ? P.wait_ns : kWaitLimitNs;

  if (tid == 0) {
    for (int s = 0; s < NST; s++) {
      mbar_init(&cs.full[s], 1);
      mbar_init(&cs.empty[s], NW);
    }
    for (int b = 0; b <= kLag; b++) {
      mbar_init(&cs.redf[b], NCT);
      mbar_init(&cs.hlf[b], 1);
    }
    mbar_fence_init();
  }
  // consumer prologue, overlapping the router's tail: the limbs of this thread's chunk of x
  const int c = tid % C, r0 = tid / C;  // consumers: r0 in {0, 1}
  Limbs X;
  if (warp < NW) {
    float xv[32];
    load_chunk_f32(P.x, P.x_dtype, 0, 32 * c, D, xv);
    if (!make_limbs(xv, X)) set_error(P.err, COLI_E_NONFINITE);
  }
  griddep_wait();  // idx, w and n_sel come from the router
  if (tid == 0) {
    int m = P.n_sel ? ld_cg_i32(P.n_sel) : P.K;
    cs.m = m < 0 ? 0 : (m > P.K ? P.K : m);
  }
  __syncthreads();
  const int m = cs.m;
  if (tid < m) {
    StreamSlot& sl = cs.slot[tid];
    const int e = ld_cg_i32(P.idx + tid);
    bool ok = e >= 0 && e < COLI_MAX_EXPERTS && P.table[e].valid;
    if (!ok) set_error(P.err, COLI_E_ROUTE);
    if (ok) {
      const TensorDesc& g = P.table[e].t[T_GATE];
      const TensorDesc& u = P.table[e].t[T_UP];
      const TensorDesc& d = P.table[e].t[T_DOWN];
      sl.gw = g.w;
      sl.uw = u.w;
      sl.dp = d.panel;
      sl.gs = g.s;
      sl.us = u.s;
      sl.gmode = g.mode;
      sl.umode = u.mode;
      sl.dmode = d.mode;
      sl.ds = d.mode == SCALE_ROW ? d.s : d.sT;
      sl.Gg = g.G;
      sl.Gu = u.G;
      sl.gsg = g.gs;
      sl.gsu = u.gs;
      sl.gsd = d.gs;
      sl.wk = ld_cg_f32(P.w + tid);
      // the host launches this kernel only for tables it can stream; anything else is a bad entry
      if (sl.gmode == SCALE_GENERIC || sl.umode == SCALE_GENERIC || sl.dmode == SCALE_GENERIC || !sl.dp ||
          !sl.ds || (sl.gmode == SCALE_CHUNK && rows_bytes + 64u * sl.Gg > SB) ||
          (sl.umode == SCALE_CHUNK && rows_bytes + 64u * sl.Gu > SB)) {
        ok = false;
        set_error(P.err, COLI_E_ROUTE);
      }
    }
    sl.ok = ok;
  }
  __syncthreads();
  griddep_launch_dependents();

  const int UB = P.I / kPanelCols;  // units per slot
  const long long total = (long long)m * UB;
  const int ubeg = (int)((long long)blockIdx.x * total / gridDim.x);
  const int uend = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);

  if (warp == NW) {
    // ---------------- producer: one lane issues every copy of this CTA's units ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      uint32_t q = 0, s = 0, ph = 0;  // stage sequence number, its slot and the slot's use parity
      bool pstop = false;
      // one stage of up to two pieces (weights, then their chunk scales) on one barrier
      auto issue = [&](const void* src, uint32_t bytes, const void* src2, uint32_t bytes2, bool weights) {
        if (pstop) return;
        if (q >= (uint32_t)NST && !mbar_wait_suspend(&cs.empty[s], ph ^ 1u, lim)) {
          pstop = true;
          set_error(P.err, COLI_E_TIMEOUT);
          return;
        }
        mbar_arrive_expect_tx(&cs.full[s], bytes + bytes2);
        uint8_t* dst = ring + (size_t)s * SB;
        if (weights)
          bulk_g2s_stream(dst, src, bytes, &cs.full[s], pol);
        else
          bulk_g2s(dst, src, bytes, &cs.full[s]);
        if (bytes2) bulk_g2s(dst + bytes, src2, bytes2, &cs.full[s]);
        q++;
        if (++s == (uint32_t)NST) {
          s = 0;
          ph ^= 1u;
        }
      };
      // the (at most kLag = 2) units whose down stages are still to come, oldest first: slot, block and
      // whether their down scales change
      int aj = 0, ab = 0, ad = 0, bj = 0, bbk = 0, bd = 0;
      auto issue_down = [&](int j, int b, int dsc) {
        const StreamSlot& sd = cs.slot[j];
        if (dsc)
          issue(sd.dmode == SCALE_CHUNK ? sd.ds + (size_t)(b * kPanelCols / sd.gsd) * D : sd.ds, 4u * D, nullptr, 0u,
                false);
        issue(sd.dp + (size_t)b * rows_bytes, rows_bytes, nullptr, 0u, true);
      };
      int prev = -1, n = 0;
      for (int u = ubeg; u < uend && !pstop; u++) {
        const int j = u / UB, b = u - j * UB;
        const StreamSlot& sl = cs.slot[j];
        if (!sl.ok) continue;
        const int i0 = b * kPanelCols;
        const bool gch = sl.gmode == SCALE_CHUNK, uch = sl.umode == SCALE_CHUNK;
        issue(sl.gw + (size_t)i0 * pitch, rows_bytes, sl.gs + (size_t)i0 * sl.Gg, gch ? 64u * sl.Gg : 0u, true);
        issue(sl.uw + (size_t)i0 * pitch, rows_bytes, sl.us + (size_t)i0 * sl.Gu, uch ? 64u * sl.Gu : 0u, true);
        const int dsc = sl.dmode == SCALE_CHUNK || j != prev;
        prev = j;
        if (n >= kLag) {  // the oldest pending unit's down stages; then shift the pending pair
          issue_down(aj, ab, ad);
          aj = bj, ab = bbk, ad = bd;
          bj = j, bbk = b, bd = dsc;
        } else if (n == 1) {
          bj = j, bbk = b, bd = dsc;
        } else {
          aj = j, ab = b, ad = dsc;
        }
        n++;
      }
      if (n >= 1) issue_down(aj, ab, ad);
      if (n >= 2) issue_down(bj, bbk, bd);
      // never leave with copies in flight into the ring
      for (uint32_t r = q > (uint32_t)NST ? q - NST : 0; r < q; r++)
        (void)mbar_wait_suspend(&cs.full[r % NST], (r / NST) & 1, lim);
    }
  } else if (warp == NW + 1) {
    // ---------------- h warp: row sums of a unit -> h = SiLU(g s_g) (u s_u) -> limbs ----------------
    bool stop = false;
    int n = 0;
    // row scales of the next kept unit's row i0 + lane (1 for chunk scales, applied per chunk), loaded
    // one unit ahead so that their latency hides behind the current unit
    int u = ubeg;
    auto next_scales = [&](float& fg, float& fu) {
      fg = fu = 1.f;
      for (; u < uend; u++) {
        const int j = u / UB;
        const StreamSlot& sl = cs.slot[j];
        if (!sl.ok) continue;
        const int i0 = (u - j * UB) * kPanelCols;
        if (lane < 16) {
          if (sl.gmode == SCALE_ROW) fg = __ldg(sl.gs + i0 + lane);
          if (sl.umode == SCALE_ROW) fu = __ldg(sl.us + i0 + lane);
        }
        u++;
        return true;
      }
      return false;
    };
    float fg, fu;
    bool have = next_scales(fg, fu);
    while (have) {
      float fg_next, fu_next;
      const bool have_next = next_scales(fg_next, fu_next);
      const int bb = n % (kLag + 1);
      const bool ok = stop || mbar_wait_suspend(&cs.redf[bb], (n / (kLag + 1)) & 1, lim);
      if (__any_sync(0xffffffffu, !ok) && !stop) {
        stop = true;
        if (lane == 0) set_error(P.err, COLI_E_TIMEOUT);
      }
      float h = 0.f;
      if (lane < 16 && !stop) {
        // row `lane` = r0 + 2 i of the unit is value i (gate) and 8 + i (up) of the warps with that r0
        const int rg = lane & 1, v = lane >> 1;
        float g = 0.f, uu = 0.f;
        for (int w = rg * (NW / 2); w < (rg + 1) * (NW / 2); w++) {
          g += cs.red[bb][w][v];
          uu += cs.red[bb][w][8 + v];
        }
        h = silu_mul(g * fg, uu * fu);
      }
      float hv[16];
#pragma unroll
      for (int i = 0; i < 16; i++) hv[i] = __shfl_sync(0xffffffffu, h, i);
      Limbs16 L;
      const bool fin = make_limbs(hv, L);
      if (lane == 0) {
        if (!fin && !stop) set_error(P.err, COLI_E_NONFINITE);
        cs.hl[bb] = L;
        mbar_arrive(&cs.hlf[bb]);
      }
      n++;
      fg = fg_next;
      fu = fu_next;
      have = have_next;
    }
  } else {
    // ---------------- consumers ----------------
    float acc[16], ws[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      acc[i] = 0.f;
      ws[i] = 0.f;
    }
    uint32_t s = 0, ph = 0;  // ring slot of the next stage and its use parity
    bool stop = false;
    auto wait_stage = [&]() -> const uint8_t* {
      if (!stop && !mbar_wait_suspend(&cs.full[s], ph, lim)) {
        stop = true;
        set_error(P.err, COLI_E_TIMEOUT);
      }
      return ring + (size_t)s * SB;
    };
    auto release_stage = [&]() {
      __syncwarp();
      if (lane == 0 && !stop) mbar_arrive(&cs.empty[s]);
      if (++s == (uint32_t)NST) {
        s = 0;
        ph ^= 1u;
      }
    };
    // the (at most kLag = 2) units whose down stages are still to come, oldest first: slot and whether
    // their down scales change
    int aj = 0, ad = 0, bj = 0, bd = 0;
    // the down part of this CTA's kept unit nn (slot j): w_k times the down scales of this thread's 16
    // rows when they change, then rows tid + jj NCT of the unit's panel, columns i0 .. i0 + 15
    auto do_down = [&](int nn, int j, int dsc) {
      const int bb = nn % (kLag + 1);
      if (dsc) {
        const float wk = cs.slot[j].wk;
        const float* sd = reinterpret_cast<const float*>(wait_stage());
#pragma unroll
        for (int jj = 0; jj < 16; jj++) ws[jj] = wk * sd[tid + jj * NCT];
        release_stage();
      }
      if (!stop && !mbar_wait_suspend(&cs.hlf[bb], (nn / (kLag + 1)) & 1, lim)) {
        stop = true;
        set_error(P.err, COLI_E_TIMEOUT);
      }
      const Limbs16 HL = cs.hl[bb];
      const uint8_t* st = wait_stage();
#pragma unroll
      for (int jj = 0; jj < 16; jj++) {
        const uint2 wv = lds64(st + (size_t)(tid + jj * NCT) * 8);
        acc[jj] = fmaf(ws[jj], chunk_dot16(wv, HL), acc[jj]);
      }
      release_stage();
    };
    int prev = -1, n = 0;
    for (int u = ubeg; u < uend; u++) {
      const int j = u / UB;
      const StreamSlot& sl = cs.slot[j];
      if (!sl.ok) continue;
      const int bb = n % (kLag + 1);
      const int dsc = sl.dmode == SCALE_CHUNK || j != prev;
      prev = j;
      // gate, then up: rows r0 + 2 i (i < 8) of the unit, this thread's chunk; chunk-group scales
      // follow the 16 rows in the stage
      float v[16];
      {
        const uint8_t* st = wait_stage();
        const float* sc = reinterpret_cast<const float*>(st + rows_bytes);
        const int gg = sl.gmode == SCALE_CHUNK ? (32 * c) / sl.gsg : 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
          v[i] = chunk_dot(lds128(st + (r0 + 2 * i) * pitch + 16 * c), X);
          if (sl.gmode == SCALE_CHUNK) v[i] *= sc[(r0 + 2 * i) * sl.Gg + gg];
        }
        release_stage();
      }
      {
        const uint8_t* st = wait_stage();
        const float* sc = reinterpret_cast<const float*>(st + rows_bytes);
        const int gu = sl.umode == SCALE_CHUNK ? (32 * c) / sl.gsu : 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
          v[8 + i] = chunk_dot(lds128(st + (r0 + 2 * i) * pitch + 16 * c), X);
          if (sl.umode == SCALE_CHUNK) v[8 + i] *= sc[(r0 + 2 * i) * sl.Gu + gu];
        }
        release_stage();
      }
      // lanes 2 i, 2 i + 1 end with the warp total of value i: gate row r0 + 2 i (i < 8) or up row
      // r0 + 2 (i - 8); the h warp takes it from here
      warp_transpose_reduce<16>(v, lane);
      if (!(lane & 1)) cs.red[bb][warp][lane >> 1] = v[0];
      mbar_arrive(&cs.redf[bb]);
      if (n >= kLag) {  // the oldest pending unit's down part; then shift the pending pair
        do_down(n - kLag, aj, ad);
        aj = bj, ad = bd;
        bj = j, bd = dsc;
      } else if (n == 1) {
        bj = j, bd = dsc;
      } else {
        aj = j, ad = dsc;
      }
      n++;
    }
    if (n >= 2) {
      do_down(n - 2, aj, ad);
      do_down(n - 1, bj, bd);
    } else if (n == 1) {
      do_down(0, aj, ad);
    }
    float* prow = P.part + (size_t)blockIdx.x * D;
#pragma unroll
    for (int jj = 0; jj < 16; jj++) prow[tid + jj * NCT] = acc[jj];
  }

  // ---------------- every CTA's partial row is stored: fixed-order reduce ----------------
  const bool arrive = !(P.withhold && blockIdx.x == 0);
  if (!grid_barrier(P.bar, lim, arrive)) {
    if (tid == 0) set_error(P.err, COLI_E_TIMEOUT);
    return;
  }
  if (!arrive) return;
  const int G = gridDim.x, nthr = blockDim.x;
  const int d0 = (int)((long long)blockIdx.x * D / G), d1 = (int)((long long)(blockIdx.x + 1) * D / G);
  const int nd = d1 - d0;
  if (nd <= 0) return;
  const int groups = max(1, min(G, nthr / nd));  // partial rows split into `groups` runs of CTAs
  const int wd = nthr / groups;                  // values of y per pass
  for (int pb = d0; pb < d1; pb += wd) {
    const int dl = tid % wd, grp = tid / wd, d = pb + dl;
    if (grp < groups) {
      float s = 0.f;
      if (d < d1) {
        const int c0 = (int)((long long)grp * G / groups), c1 = (int)((long long)(grp + 1) * G / groups);
#pragma unroll 8
        for (int cc = c0; cc < c1; cc++) s += __ldcg(P.part + (size_t)cc * D + d);
      }
      cs.fold[grp * wd + dl] = s;
    }
    __syncthreads();
    if (tid < wd && pb + tid < d1) {
      const int dd = pb + tid;
      float tot = 0.f;
      for (int g2 = 0; g2 < groups; g2++) tot += cs.fold[g2 * wd + tid];
      if (P.resid) tot = load_act(P.resid, P.x_dtype, dd) + tot;
      if (P.y_dtype == COLI_DTYPE_F32)
        static_cast<float*>(P.y)[dd] = tot;
      else
        static_cast<uint16_t*>(P.y)[dd] = f32_to_bf16_rn(tot);
    }
    __syncthreads();
  }
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

bool stream_eligible(const coli_ctx* ctx, int S) {
  const int D = ctx->table_D, I = ctx->table_I;
  return S == 1 && ctx->stream_ffn && !ctx->decode_fused && ctx->coop_mode > 0 && ctx->table_count > 0 &&
         ctx->table_nostream == 0 && D % 1024 == 0 && D <= 512 * kStMaxWarps && I % kPanelCols == 0;
}

int launch_stream_ffn(coli_ctx* ctx, const void* x, int x_dtype, const int32_t* idx, const float* w,
                      const int32_t* n_sel, int K, const void* resid, void* y, int y_dtype) {
  const int D = ctx->table_D, I = ctx->table_I;
  const int NW = D / 512, threads = 32 * (NW + 2);
  // a unit's 16 gate (or up) rows and their chunk-group scales; the down panel and down scales are smaller
  const uint32_t SB = (uint32_t)align_up(8u * (uint32_t)D + 64u * (uint32_t)ctx->table_gu_maxG, 128);
  int maxsm = 0;
  cudaError_t e = cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream FFN: shared memory limit");
  const long long room = (long long)maxsm - 128 - (long long)stream_ctrl_bytes();
  int nst = (int)(room / SB);
  if (nst > kStMaxStages) nst = kStMaxStages;
  if (nst < kStMinStages) return fail(ctx, COLI_E_INVAL, "stream FFN: not enough shared memory for the ring");
  const size_t smem = 128 + stream_ctrl_bytes() + (size_t)nst * SB;
  auto kern = threads <= 320 ? stream_ffn_kernel<320> : (threads <= 448 ? stream_ffn_kernel<448> : stream_ffn_kernel<576>);
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return cuda_fail(ctx, e, "stream FFN: shared memory attribute");
  int occ = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem)) != cudaSuccess || occ < 1)
    return e != cudaSuccess ? cuda_fail(ctx, e, "stream FFN: occupancy") : fail(ctx, COLI_E_CUDA, "stream FFN: no residency");
  const int G = ctx->num_sms;
  int rc = ensure_workspace(ctx, (size_t)G * D * sizeof(float));
  if (rc != COLI_OK) return rc;
  StreamParams P;
  P.x = x;
  P.x_dtype = x_dtype;
  P.y_dtype = y_dtype;
  P.D = D;
  P.I = I;
  P.K = K;
  P.idx = idx;
  P.w = w;
  P.n_sel = n_sel;
  P.table = ctx->d_table;
  P.resid = resid;
  P.y = y;
  P.part = reinterpret_cast<float*>(ctx->ws.base);
  P.bar = reinterpret_cast<unsigned long long*>(ctx->d_status + kStreamBar);
  P.err = ctx->d_status;
  P.nst = nst;
  P.sb = SB;
  P.wait_ns = ctx->wait_ns;
  P.withhold = ctx->test_withhold > 0;  // one-shot: only the next launch withholds
  if (ctx->test_withhold > 0) ctx->test_withhold--;
  ProfScope prof(ctx, COLI_KERNEL_GATEUP);
  e = launch_k(kern, G, threads, smem, ctx->stream, ctx->coop_mode == 2, true, P);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream FFN launch");
  return COLI_OK;
}

}  // namespace coli
