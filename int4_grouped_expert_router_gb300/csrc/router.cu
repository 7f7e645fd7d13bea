// Device router: f32 logits GEMV + sigmoid + bias, then bias-augmented top-K selection, raw-score
// weights, top-p, norm_topk and routed_scale.
//
// c/backend_cuda.cu commit history, commit "First increment of the #431 plan": an E x D f32
// logits GEMV + sigmoid, then a selection step that does bias-augmented top-K by choice with a
// strict '>' tie-break, weights from the raw score, route-level TOPP truncation, norm_topk and
// routed_scale. For S > 1 the logits of all tokens come from one launch (the batched router of
// the "GPU resident pipeline" commit).
#include <algorithm>
#include <mutex>
#include <string>

#include "coli_internal.h"
#include "pipe.h"

namespace coli {

constexpr int kRouterThreads = 256;
// Fewer tokens than kBatchedS take the one-launch router below; more take the tiled-GEMM router.
constexpr int kBatchedS = 16;
// The one-launch router's selection holds at most 32 experts per lane (E <= 1024); larger E
// takes the many-token path, whose separate selection kernel also has the large-E form.
constexpr int kDecodeMaxE = 1024;
constexpr int kRouterMaxParts = 4;  // column parts of a logit row
// Router scratch of a context (and of the no-allocation entry): the launch counter in the first
// 256 bytes, then one 64-bit word per (token, column part, expert).
constexpr size_t kRouterWordsOff = 256;
static_assert(kRouterScratchBytes >= kRouterWordsOff + (size_t)(kBatchedS - 1) * kDecodeMaxE * 8,
              "router scratch holds S < kBatchedS tokens of P x E <= kDecodeMaxE words");

// Order-preserving map of a finite binary32 value to uint32 (larger float -> larger integer;
// -0 is folded onto +0 so that the two compare equal, as floats do). Every finite value maps to
// at least 0x00800000, so 0 marks an absent expert.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (no memory clobber: a poll issues all of its loads before it looks at any result)
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// "a ranks before b": a larger choice key, or an equal key and a lower expert index.
__device__ __forceinline__ bool ranks_before(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// A lane's N candidates (key, slot i, raw score) sorted into ranking order by a bitonic network
// (all indices compile-time, so the arrays stay in registers). Slot i is expert lane + 32 i, so
// comparing slots compares expert indices.
template <int N>
__device__ __forceinline__ void sort_lane(uint32_t (&k)[N], int (&ii)[N], float (&s)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < N; i++) {
        const int j = i ^ stride;
        if (j > i) {
          const bool first_is_i = ranks_before(k[i], ii[i], k[j], ii[j]);
          const bool swap = ((i & size) == 0) ? !first_is_i : first_is_i;
          if (swap) {
            const uint32_t tk = k[i];
            k[i] = k[j];
            k[j] = tk;
            const int ti = ii[i];
            ii[i] = ii[j];
            ii[j] = ti;
            const float ts = s[i];
            s[i] = s[j];
            s[j] = ts;
          }
        }
      }
    }
  }
}

// Lane k holds the expert of slot k (mine) and its raw score (wmine): weights from the raw
// (bias-free) score, top-p, norm and scale; every sum in slot order in binary32, no contraction.
// The K scores reach every lane through independent shuffles, so only the additions form a chain.
template <int KMAX>
__device__ __forceinline__ void select_finish(int mine, float wmine, int K, float topp, int norm_topk,
                                              float routed_scale, int shared, int32_t* __restrict__ idx_out,
                                              float* __restrict__ w_out, int32_t* __restrict__ nsel_out,
                                              const ExpertDesc* table) {
  const int lane = threadIdx.x & 31;
  float pre[KMAX];  // pre[k]: the slot-order sum of scores 0..k
  float total = 0.f;
#pragma unroll
  for (int k = 0; k < KMAX; k++) {
    const float v = __shfl_sync(0xffffffffu, wmine, k);
    if (k < K) total = __fadd_rn(total, v);
    pre[k] = total;
  }
  int m = K;
  if (topp > 0.f && topp < 1.f) {
    const float q = __fdiv_rn(wmine, total);  // lane k: the share of slot k
    float cum = 0.f;
    bool done = false;
#pragma unroll
    for (int k = 0; k < KMAX; k++) {
      const float qk = __shfl_sync(0xffffffffu, q, k);
      if (k < K && !done) {
        cum = __fadd_rn(cum, qk);
        if (cum >= topp) {
          m = k + 1;
          done = true;
        }
      }
    }
  }
  float denom = 1.f;
  if (norm_topk) {
#pragma unroll
    for (int k = 0; k < KMAX; k++)
      if (k == m - 1) denom = pre[k];
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

// One warp selects for one token from its lanes' candidates (lane l holds experts l + 32 i, i <
// EPL, as choice keys, slots and raw scores; absent experts have key 0). Each lane sorts its own
// candidates once; every round then compares only the lanes' heads: the largest key, and among the
// lanes holding it (rarely more than one) the lowest expert index, wins; the winner's lane pops its
// head. Ties therefore go to the lower index, as a strict '>' scan in increasing index order gives.
// With more than 8 experts per lane (E > 256) the lane does not sort (a 16- or 32-element network
// costs more than it saves); each round it scans its not-yet-chosen candidates in increasing index
// order with a strict '>' instead, which yields the same head.
template <int EPL, int KMAX>
__device__ __forceinline__ void select_sorted(uint32_t (&key)[EPL], int (&ii)[EPL], float (&sv)[EPL], int K,
                                              float topp, int norm_topk, float routed_scale, int shared,
                                              int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                              int32_t* __restrict__ nsel_out, const ExpertDesc* table) {
  const int lane = threadIdx.x & 31;
  constexpr bool kSort = EPL <= 8;
  if constexpr (kSort) sort_lane<EPL>(key, ii, sv);
  int mine = -1;      // lane k keeps the expert chosen in round k ...
  float wmine = 0.f;  // ... and its raw score
  for (int k = 0; k < K; k++) {
    uint32_t hk = key[0];
    int hi = 0;  // position of the lane's head (always 0 when sorted)
    if constexpr (!kSort) {
#pragma unroll
      for (int i = 1; i < EPL; i++)
        if (key[i] > hk) {
          hk = key[i];
          hi = i;
        }
    }
    const int he = lane + 32 * (kSort ? ii[0] : hi);
    const uint32_t best = __reduce_max_sync(0xffffffffu, hk);
    const unsigned tied = __ballot_sync(0xffffffffu, hk == best);
    int wl;
    if (__popc(tied) == 1) {
      wl = __ffs(tied) - 1;
    } else {
      wl = (int)(__reduce_min_sync(0xffffffffu, hk == best ? (uint32_t)he : 0xffffffffu) & 31u);
    }
    float hs = sv[0];
    if constexpr (!kSort) {
#pragma unroll
      for (int i = 1; i < EPL; i++)
        if (i == hi) hs = sv[i];
    }
    const int we = __shfl_sync(0xffffffffu, he, wl);
    const float ws = __shfl_sync(0xffffffffu, hs, wl);
    if (lane == k) {
      mine = we;
      wmine = ws;
    }
    if (lane == wl) {
      if constexpr (kSort) {
#pragma unroll
        for (int i = 0; i + 1 < EPL; i++) {
          key[i] = key[i + 1];
          ii[i] = ii[i + 1];
          sv[i] = sv[i + 1];
        }
        key[EPL - 1] = 0u;
      } else {
#pragma unroll
        for (int i = 0; i < EPL; i++)
          if (i == hi) key[i] = 0u;  // chosen: below every candidate
      }
    }
  }
  select_finish<KMAX>(mine, wmine, K, topp, norm_topk, routed_scale, shared, idx_out, w_out, nsel_out, table);
}

// Selection of one token from its (score, choice) pairs in memory (the many-token path).
template <int EPL, int KMAX>
__device__ __forceinline__ void select_pairs(const float2* __restrict__ sc_row, int E, int K, float topp, int norm_topk,
                                             float routed_scale, int shared, int32_t* __restrict__ idx_out,
                                             float* __restrict__ w_out, int32_t* __restrict__ nsel_out, int* err,
                                             const ExpertDesc* table) {
  const int lane = threadIdx.x & 31;
  uint32_t key[EPL];
  int ii[EPL];
  float sv[EPL];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < EPL; i++) {
    const int e = lane + 32 * i;
    ii[i] = i;
    if (e < E) {
      const float2 v = __ldcg(sc_row + e);  // (score, choice)
      if (!isfinite(v.x) || !isfinite(v.y)) bad = true;
      key[i] = order_key(v.y);
      sv[i] = v.x;
    } else {
      key[i] = 0u;
      sv[i] = 0.f;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, COLI_E_NONFINITE);
  select_sorted<EPL, KMAX>(key, ii, sv, K, topp, norm_topk, routed_scale, shared, idx_out, w_out, nsel_out, table);
}

// Selection for 1024 < E <= COLI_MAX_EXPERTS (more than 32 experts per lane): the same ranking
// rule, but each round re-reads the lane's (score, choice) pairs through L2 instead of holding
// them in registers, and the chosen set is a 128-bit mask per lane.
__device__ void select_pairs_large(const float2* __restrict__ sc_row, int E, int K, float topp, int norm_topk,
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
  select_finish<32>(mine, wmine, K, topp, norm_topk, routed_scale, shared, idx_out, w_out, nsel_out, table);
}

// ------------------------------------------------------------------------------------------
// Fewer than kBatchedS tokens: one launch. CTA b computes R rows (experts) of the logits over one
// of P column parts of D for every token and publishes each partial sum as one 64-bit word: its
// binary32 bits in the low half and this launch's tag (the scratch's launch counter plus one) in
// the high half. A single 64-bit store is single-copy atomic, so a reader that sees the tag sees
// the value, and no fence or arrival counter stands between a CTA's last FMA and the selection.
// CTA 0, after its own rows, polls every word of a token (one warp per token) until all carry the
// tag -- a wait bounded by the context's limit, after which it records COLI_E_TIMEOUT and writes
// an empty route -- then sums each expert's P partials in part order, applies the sigmoid and the
// bias, selects, and at the end advances the counter. Tags only grow, so a word left by an earlier
// launch (or by one that gave up) never matches a later launch's tag.
//
// Ordering between launches: every CTA reads the counter after griddepcontrol.wait, which returns
// only once the preceding kernel in the stream (and, through its own wait, every kernel before it)
// has completed, so the previous launch's advance is visible; within a launch the advance comes
// after every CTA has published, hence after every CTA has read the counter.
// ------------------------------------------------------------------------------------------

struct RouterArgs {
  const void* x;
  const float* Wr;
  const float* bias;
  int32_t* idx;
  float* w;
  int32_t* n_sel;
  int* err;
  const ExpertDesc* table;
  unsigned* counter;         // launch counter (its 64-bit words follow at kRouterWordsOff)
  unsigned long long* words; // [S][P][E] tagged partial logits
  unsigned long long wait_ns;
  int x_dtype, S, D, E, K;
  float topp;
  int norm_topk;
  float routed_scale;
  int shared;
  int parts, part_cols;      // P and the columns of each part (a multiple of 4)
  int withhold;              // test hook: the last CTA does not publish token 0
};

constexpr int kSelBatch = 4;  // tokens whose keys CTA 0 holds in shared memory at a time

// Weights of one token's selection (every lane of the warp runs it; lane k holds slot k's expert
// `mine` and raw score `wmine`): weights from the raw (bias-free) score, top-p, norm and scale,
// every sum in slot order in binary32, no contraction. The loops are rolled: this code runs once
// per launch, usually with a cold instruction cache, so its length costs more than its latency.
__device__ __forceinline__ void finish_rolled(int mine, float wmine, int K, float topp, int norm_topk,
                                              float routed_scale, int shared, int32_t* __restrict__ idx_out,
                                              float* __restrict__ w_out, int32_t* __restrict__ nsel_out,
                                              const ExpertDesc* table) {
  const int lane = threadIdx.x & 31;
  int m = K;
  float total = 0.f;
  for (int k = 0; k < K; k++) total = __fadd_rn(total, __shfl_sync(0xffffffffu, wmine, k));
  if (topp > 0.f && topp < 1.f) {
    const float q = __fdiv_rn(wmine, total);  // lane k: the share of slot k
    float cum = 0.f;
    for (int k = 0; k < K; k++) {  // every lane sees the same sums, so the exit is uniform
      cum = __fadd_rn(cum, __shfl_sync(0xffffffffu, q, k));
      if (cum >= topp) {
        m = k + 1;
        break;
      }
    }
  }
  float denom = 1.f;
  if (norm_topk) {
    denom = 0.f;
    for (int k = 0; k < m; k++) denom = __fadd_rn(denom, __shfl_sync(0xffffffffu, wmine, k));
  }
  const bool has_shared = shared >= 0;
  if (lane < K + has_shared) {
    const bool kept = lane < m;
    const bool is_shared = has_shared && lane == m;
    const float wv = norm_topk ? __fdiv_rn(wmine, denom) : wmine;
    idx_out[lane] = kept ? mine : (is_shared ? shared : -1);
    w_out[lane] = kept ? __fmul_rn(wv, routed_scale) : (is_shared ? 1.0f : 0.f);
  }
  if (lane == 0 && nsel_out) *nsel_out = m + has_shared;
  const int pe = lane < K ? mine : (has_shared && lane == K ? shared : -1);
  if (table && pe >= 0)
    for (int l = 0; l < (int)(sizeof(ExpertDesc) / 128); l++)
      prefetch_l2_line(reinterpret_cast<const char*>(table + pe) + 128 * l);
}

// CTA 0's selection of every token, kSelBatch tokens at a time. Each thread takes (token, expert)
// items: it polls the item's P words until all carry the tag (all P loads in flight per poll; a
// wait bounded by `limit`), sums them in part order, applies the sigmoid and the bias and stores
// the choice key and the raw score in shared memory. Warp w then selects token w of the batch
// with K rounds over the keys: each lane scans its experts (lane, lane + 32, ...) with a strict
// '>', the warp takes the largest key and, among the lanes holding it, the lowest index; the
// winner's key is zeroed (every finite choice maps to a nonzero key). A token with a word that
// never arrived gets COLI_E_TIMEOUT and an empty route.
__device__ __forceinline__ void select_tokens(const RouterArgs& a, unsigned tag) {
  // keys [nbmax][E] then raw scores [nbmax][E] in dynamic shared memory, nbmax = min(S, kSelBatch):
  // every CTA of the grid gets the allocation, so it is kept to what CTA 0 needs (2 KiB for one token
  // of 256 experts) and does not stop the expert kernel's CTAs from sharing the SMs
  extern __shared__ uint32_t router_dyn[];
  __shared__ int s_late[kSelBatch];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, P = a.parts;
  const int nbmax = min(a.S, kSelBatch);
  uint32_t* skey = router_dyn;
  float* ssc = reinterpret_cast<float*>(router_dyn + (size_t)nbmax * E);
  const uint64_t limit = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  const int slots = a.K + (a.shared >= 0);
  for (int t0 = 0; t0 < a.S; t0 += kSelBatch) {
    const int nb = min(kSelBatch, a.S - t0);
    if (tid < kSelBatch) s_late[tid] = 0;
    __syncthreads();
    bool bad = false;
    for (int it = tid; it < nb * E; it += kRouterThreads) {
      const int tb = it / E, e = it - tb * E;
      const unsigned long long* wp = a.words + (size_t)(t0 + tb) * P * E + e;
      float z[kRouterMaxParts] = {0.f, 0.f, 0.f, 0.f};
      bool late = false;
      const uint64_t t_start = globaltimer_ns();
      for (;;) {
        unsigned long long v[kRouterMaxParts];
#pragma unroll
        for (int p = 0; p < kRouterMaxParts; p++) v[p] = p < P ? ld_relaxed_u64(wp + (size_t)p * E) : 0ull;
        bool ready = true;
#pragma unroll
        for (int p = 0; p < kRouterMaxParts; p++) {
          z[p] = __uint_as_float((unsigned)v[p]);
          if (p < P && (unsigned)(v[p] >> 32) != tag) ready = false;
        }
        if (ready) break;
        if (globaltimer_ns() - t_start > limit) {
          late = true;
          s_late[tb] = 1;
          break;
        }
      }
      float zs = z[0];
#pragma unroll
      for (int p = 1; p < kRouterMaxParts; p++)
        if (p < P) zs = __fadd_rn(zs, z[p]);
      const float sc = 1.0f / (1.0f + expf(-zs));
      const float ch = a.bias ? __fadd_rn(sc, __ldg(a.bias + e)) : sc;
      if (!late && (!isfinite(sc) || !isfinite(ch))) bad = true;
      skey[tb * E + e] = order_key(ch);
      ssc[tb * E + e] = sc;
    }
    if (bad) set_error(a.err, COLI_E_NONFINITE);
    __syncthreads();
    if (warp < nb) {
      const int t = t0 + warp;
      int32_t* io = a.idx + (size_t)t * slots;
      float* wo = a.w + (size_t)t * slots;
      int32_t* no = a.n_sel ? a.n_sel + t : nullptr;
      if (s_late[warp]) {
        if (lane == 0) set_error(a.err, COLI_E_TIMEOUT);
        if (lane < slots) {
          io[lane] = -1;
          wo[lane] = 0.f;
        }
        if (lane == 0 && no) *no = 0;
      } else {
        uint32_t* kw = skey + warp * E;
        int mine = -1;
        float wmine = 0.f;
        for (int k = 0; k < a.K; k++) {
          uint32_t bk = 0u;
          int be = 0;
          for (int e = lane; e < E; e += 32) {
            const uint32_t key = kw[e];
            if (key > bk) {
              bk = key;
              be = e;
            }
          }
          const uint32_t best = __reduce_max_sync(0xffffffffu, bk);
          const uint32_t win = __reduce_min_sync(0xffffffffu, bk == best ? (uint32_t)be : 0xffffffffu);
          if (lane == (int)(win & 31u)) kw[win] = 0u;
          __syncwarp();
          if (lane == k) {
            mine = (int)win;
            wmine = ssc[warp * E + win];
          }
        }
        finish_rolled(mine, wmine, a.K, a.topp, a.norm_topk, a.routed_scale, a.shared, io, wo, no, a.table);
      }
    }
    __syncthreads();  // before the next batch reuses the keys
  }
}

// Partial logits of R rows over the columns [c0, c1) of one token. XT: 0 f32 activations and
// 16-byte aligned rows (float4 loads), 1 bf16 activations 8-byte aligned (4 per load), 2 any
// layout (one element per load). NV vector loads per row are in flight per thread at a time:
// with D = 6144 and up to 8 * 256 * 4 columns per part, every load of a thread issues before the
// first FMA, so the row costs one memory round trip.
template <int XT, int R>
__device__ __forceinline__ void router_rows(const RouterArgs& a, int t, int e0, int nrows, int c0, int c1,
                                            float (&acc)[R]) {
  constexpr int NV = R == 1 ? 8 : (R == 2 ? 4 : 2);
  const int tid = threadIdx.x;
#pragma unroll
  for (int r = 0; r < R; r++) acc[r] = 0.f;
  if constexpr (XT == 2) {
#pragma unroll 4
    for (int j = c0 + tid; j < c1; j += kRouterThreads) {
      const float b = load_act(a.x, a.x_dtype, (size_t)t * a.D + j);
#pragma unroll
      for (int r = 0; r < R; r++)
        if (r < nrows) acc[r] = fmaf(__ldg(a.Wr + (size_t)(e0 + r) * a.D + j), b, acc[r]);
    }
  } else {
    const int j1 = c1 >> 2;
    for (int jb = (c0 >> 2) + tid; jb < j1; jb += NV * kRouterThreads) {
      float4 xv[NV], wv[R][NV];
#pragma unroll
      for (int v = 0; v < NV; v++) {
        const int j = jb + v * kRouterThreads;
        if (j < j1) {
          if constexpr (XT == 0) {
            xv[v] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)t * a.D) + j);
          } else {
            const uint2 h = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.x) +
                                                                 (size_t)t * a.D) + j);
            xv[v] = make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xffff0000u),
                                __uint_as_float(h.y << 16), __uint_as_float(h.y & 0xffff0000u));
          }
#pragma unroll
          for (int r = 0; r < R; r++)
            wv[r][v] = r < nrows ? __ldg(reinterpret_cast<const float4*>(a.Wr + (size_t)(e0 + r) * a.D) + j)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          xv[v] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int r = 0; r < R; r++) wv[r][v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int v = 0; v < NV; v++)
#pragma unroll
        for (int r = 0; r < R; r++) {
          acc[r] = fmaf(wv[r][v].x, xv[v].x, acc[r]);
          acc[r] = fmaf(wv[r][v].y, xv[v].y, acc[r]);
          acc[r] = fmaf(wv[r][v].z, xv[v].z, acc[r]);
          acc[r] = fmaf(wv[r][v].w, xv[v].w, acc[r]);
        }
    }
  }
}

template <int XT, int R>
__global__ void __launch_bounds__(kRouterThreads) router_decode_kernel(const __grid_constant__ RouterArgs a) {
  __shared__ float red[kRouterThreads / 32][R];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p = blockIdx.x % a.parts;
  const int e0 = (blockIdx.x / a.parts) * R;
  const int nrows = min(R, a.E - e0);
  const int c0 = p * a.part_cols, c1 = min(a.D, c0 + a.part_cols);
  griddep_wait();               // x may be the previous kernel's output
  griddep_launch_dependents();  // the expert kernel may start its prologue
  const unsigned tag = ld_relaxed_u32(a.counter) + 1u;
  const bool withhold = a.withhold && blockIdx.x == gridDim.x - 1;
  for (int t = 0; t < a.S; t++) {
    float acc[R];
    router_rows<XT, R>(a, t, e0, nrows, c0, c1, acc);
#pragma unroll
    for (int r = 0; r < R; r++) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
      if (lane == 0) red[warp][r] = acc[r];
    }
    __syncthreads();
    if (tid < nrows && !(withhold && t == 0)) {
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < kRouterThreads / 32; i++) z += red[i][tid];
      st_relaxed_u64(a.words + ((size_t)t * a.parts + p) * a.E + e0 + tid,
                     ((unsigned long long)tag << 32) | __float_as_uint(z));
    }
    __syncthreads();
  }
  if (blockIdx.x != 0) return;
  select_tokens(a, tag);
  if (tid == 0) st_relaxed_u32(a.counter, tag);
}

// ------------------------------------------------------------------------------------------
// Many tokens (S >= kBatchedS): the logits as a tiled f32 GEMM, each CTA a 64-token x 64-expert
// tile over one of kRSplit column ranges of D; the ranges are summed in a fixed order, then
// sigmoid and bias give the (score, choice) pairs and one warp per token selects.
// ------------------------------------------------------------------------------------------

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

template <int EPL, int KMAX>
__global__ void router_select_kernel(const float2* sc, int S, int E, int K, float topp, int norm_topk,
                                     float routed_scale, int shared, int32_t* idx, float* w, int32_t* n_sel, int* err,
                                     const ExpertDesc* table) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= S) return;  // uniform per warp
  const int slots = K + (shared >= 0);  // output slots per token
  const float2* row = sc + (size_t)t * E;
  int32_t* io = idx + (size_t)t * slots;
  float* wo = w + (size_t)t * slots;
  int32_t* no = n_sel ? n_sel + t : nullptr;
  if constexpr (EPL == 0)
    select_pairs_large(row, E, K, topp, norm_topk, routed_scale, shared, io, wo, no, err, table);
  else
    select_pairs<EPL, KMAX>(row, E, K, topp, norm_topk, routed_scale, shared, io, wo, no, err, table);
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
  const bool k8 = K <= 8;
  switch (epl) {
#define COLI_SELECT_CASE(N)                                                                                          \
  case N:                                                                                                            \
    if (k8)                                                                                                          \
      router_select_kernel<N, 8><<<sg, 256, 0, ctx->stream>>>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared, \
                                                              idx, w, n_sel, ctx->d_status, table);                  \
    else                                                                                                             \
      router_select_kernel<N, 32><<<sg, 256, 0, ctx->stream>>>(sc_ws, S, E, K, topp, norm_topk, routed_scale,        \
                                                               shared, idx, w, n_sel, ctx->d_status, table);         \
    break;
    COLI_SELECT_CASE(1)
    COLI_SELECT_CASE(2)
    COLI_SELECT_CASE(4)
    COLI_SELECT_CASE(8)
    COLI_SELECT_CASE(16)
    COLI_SELECT_CASE(32)
    default:  // more than 1024 experts
      router_select_kernel<0, 32><<<sg, 256, 0, ctx->stream>>>(sc_ws, S, E, K, topp, norm_topk, routed_scale, shared,
                                                                idx, w, n_sel, ctx->d_status, table);
#undef COLI_SELECT_CASE
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "batched router launch");
  return COLI_OK;
}

// The one-launch router's shape: R rows per CTA and P column parts, so that about two CTAs run on
// every SM and each CTA's loads issue together (COLI_ROUTER_ROWS / COLI_ROUTER_PARTS, read at
// coli_init, override the choice). P x E never exceeds kDecodeMaxE, which bounds the words of a
// token.
struct RouterShape {
  int rows, parts, part_cols, grid;
};

static RouterShape router_shape(const coli_ctx* ctx, int E, int D, bool vec) {
  const int pmax = std::max(1, std::min(kRouterMaxParts, kDecodeMaxE / E));
  RouterShape s;
  s.rows = ctx->router_rows > 0 ? ctx->router_rows : 4;
  const int blocks = (E + s.rows - 1) / s.rows;
  int P = ctx->router_parts > 0 ? ctx->router_parts : (2 * ctx->num_sms) / blocks;
  P = std::max(1, std::min(P, pmax));
  const int q = vec ? 4 : 1;  // vector loads need parts on 4-column boundaries
  s.part_cols = ((D + P - 1) / P + q - 1) / q * q;
  s.parts = (D + s.part_cols - 1) / s.part_cols;  // no empty part
  s.grid = blocks * s.parts;
  return s;
}

template <int XT, int R>
static cudaError_t launch_decode(const cudaLaunchConfig_t* cfg, const RouterArgs& a) {
  return cudaLaunchKernelEx(cfg, router_decode_kernel<XT, R>, a);
}

template <int XT>
static cudaError_t launch_decode_rows(const cudaLaunchConfig_t* cfg, int rows, const RouterArgs& a) {
  switch (rows) {
    case 1: return launch_decode<XT, 1>(cfg, a);
    case 2: return launch_decode<XT, 2>(cfg, a);
    case 8: return launch_decode<XT, 8>(cfg, a);
    default: return launch_decode<XT, 4>(cfg, a);
  }
}

// One-launch router (S < kBatchedS, E <= kDecodeMaxE) on the scratch at `scratch` (the launch
// counter, then kRouterWordsBytes of words).
static int launch_router_decode(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                                const float* bias, int E, int K, float topp, int norm_topk, float routed_scale,
                                int shared, int32_t* idx, float* w, int32_t* n_sel, unsigned char* scratch,
                                const char* what) {
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), wa = reinterpret_cast<uintptr_t>(Wr);
  const bool rows16 = D % 4 == 0 && (wa & 15) == 0;
  const int xt = (rows16 && x_dtype == COLI_DTYPE_F32 && (xa & 15) == 0)   ? 0
                 : (rows16 && x_dtype == COLI_DTYPE_BF16 && (xa & 7) == 0) ? 1
                                                                            : 2;
  const RouterShape sh = router_shape(ctx, E, D, xt != 2);
  RouterArgs a;
  a.x = x;
  a.Wr = Wr;
  a.bias = bias;
  a.idx = idx;
  a.w = w;
  a.n_sel = n_sel;
  a.err = ctx->d_status;
  a.table = ctx->table_count > 0 ? ctx->d_table : nullptr;  // for the L2 prefetch hint
  a.counter = reinterpret_cast<unsigned*>(scratch);
  a.words = reinterpret_cast<unsigned long long*>(scratch + kRouterWordsOff);
  a.wait_ns = ctx->wait_ns;
  a.x_dtype = x_dtype;
  a.S = S;
  a.D = D;
  a.E = E;
  a.K = K;
  a.topp = topp;
  a.norm_topk = norm_topk;
  a.routed_scale = routed_scale;
  a.shared = shared;
  a.parts = sh.parts;
  a.part_cols = sh.part_cols;
  a.withhold = ctx->test_withhold_router > 0;  // one-shot: only the next launch withholds
  if (ctx->test_withhold_router > 0) ctx->test_withhold_router--;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sh.grid);
  cfg.blockDim = dim3(kRouterThreads);
  cfg.dynamicSmemBytes = (size_t)std::min(S, kSelBatch) * E * 2 * sizeof(uint32_t);  // <= 32 KiB
  cfg.stream = ctx->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope prof(ctx, COLI_KERNEL_ROUTER);
  cudaError_t e = xt == 0   ? launch_decode_rows<0>(&cfg, sh.rows, a)
                  : xt == 1 ? launch_decode_rows<1>(&cfg, sh.rows, a)
                            : launch_decode_rows<2>(&cfg, sh.rows, a);
  if (e != cudaSuccess) return cuda_fail(ctx, e, what);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, what);
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
  return launch_router_decode(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, idx, w,
                              n_sel, static_cast<unsigned char*>(ctx->d_router), "router launch");
}

// ------------------------------------------------------------------------------------------
// Router entry that allocates nothing (coli_router_select_noalloc).
//
// Some callers cannot let a call allocate device memory: a server that has handed all free HBM to
// its own caching pool (a cudaMalloc would fail or force it to evict), or a decode loop that must
// not stall, since cudaMalloc may synchronise the device and a workspace that grows waits for the
// context's stream first. This entry therefore keeps its scratch in a fixed file-scope device
// array instead of the context's workspace: the one-launch router's counter and words (as in a
// context's own router scratch), then the (score, choice) pairs of at most kFixedRouterCells
// (token, expert) cells and the partial logits of the many-token path. Its address is looked up
// once per device and CUDA context (the first call there), since a device reset or another context
// loads the module at a new address. The counter only grows, so the array needs no clearing
// between calls. All contexts on a device share the array, so calls whose kernels could overlap
// (different streams, contexts or host threads without ordering) race on it.
// ------------------------------------------------------------------------------------------

constexpr int kFixedRouterCells = 65536;  // S * E limit
constexpr int kFixedMaxDevices = 64;
// one-launch router scratch, pairs (512 KiB), partial logits of the many-token path (2 MiB)
constexpr size_t kFixedPairsOff = align_up(kRouterScratchBytes, 256);
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
  if (S >= kBatchedS || E > kDecodeMaxE)  // the many-token path, as coli_router_select takes it
    return launch_router_batched(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel,
                                 reinterpret_cast<float2*>(base + kFixedPairsOff),
                                 reinterpret_cast<float*>(base + kFixedPartOff));
  return launch_router_decode(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel,
                              base, "router_select_noalloc launch");
}

}  // namespace coli

