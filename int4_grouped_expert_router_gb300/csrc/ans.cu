// Compressed expert tier, the codec: a byte stream of packed int4 weights is split into 4 KiB blocks
// that decode independently (PR #651 "cuda: add experimental lossless compressed expert tier" keeps its
// experts as independently decodable 4096-byte ANS blocks). This codec is our own rANS over the nibbles.
//
// Format of a compressed stream (all little-endian, every section 4-byte aligned):
//   u32 magic 'C4A1' | u32 block bytes (4096) | u64 raw bytes n | u32 blocks B | u32 reserved
//   u16 freq[16]                 nibble frequencies, each >= 1, summing to 4096 (12-bit probabilities)
//   u32 offset[B + 1]            byte offset of each block from the start of the block area; offset[B] = end
//   blocks: for each block, u32 state[32] | u16 words[32] | the 32 lanes' 16-bit word streams, lane 0 first
//           (padded to 4 bytes)
// Within a block of m bytes the nibble stream is low nibble then high nibble of each byte (2m symbols);
// lane l codes symbols l, l + 32, l + 64, ... with its own rANS state (32-bit, renormalised to
// [2^16, 2^32) with 16-bit words), so a warp decodes a block with one lane per state.
#include <string.h>

#include <map>
#include <mutex>
#include <vector>

#include "ans.h"

namespace coli {

namespace {

constexpr uint32_t kMagic = 0x31413443u;  // "C4A1"
constexpr int kProbBits = 12;
constexpr uint32_t kProbScale = 1u << kProbBits;
constexpr uint32_t kLow = 1u << 16;  // lower end of the normalised state interval

struct Header {
  uint32_t magic, block_bytes;
  uint64_t n;
  uint32_t blocks, reserved;
  uint16_t freq[16];
};
static_assert(sizeof(Header) == 56, "header layout");

inline size_t align4(size_t v) { return (v + 3) & ~size_t(3); }

// 16 frequencies summing to kProbScale, each >= 1, proportional to the counts (largest remainder).
void make_freq(const uint64_t (&count)[16], uint64_t total, uint16_t (&freq)[16]) {
  uint32_t f[16];
  uint32_t sum = 0;
  for (int s = 0; s < 16; s++) {
    uint64_t v = total ? count[s] * (kProbScale - 16) / total : (kProbScale - 16) / 16;
    f[s] = (uint32_t)v + 1;
    sum += f[s];
  }
  // hand the remainder to the most frequent symbols, one each, lowest symbol first among equals
  while (sum < kProbScale) {
    int best = 0;
    for (int s = 1; s < 16; s++)
      if (count[s] > count[best]) best = s;
    for (int s = 0; s < 16 && sum < kProbScale; s++)
      if (count[s] == count[best]) {
        f[s]++;
        sum++;
      }
  }
  for (int s = 0; s < 16; s++) freq[s] = (uint16_t)f[s];
}

}  // namespace

int ans_encode(const uint8_t* in, uint64_t n, std::vector<uint8_t>& out) {
  uint64_t count[16] = {0};
  for (uint64_t i = 0; i < n; i++) {
    count[in[i] & 15]++;
    count[in[i] >> 4]++;
  }
  Header h{};
  h.magic = kMagic;
  h.block_bytes = kAnsBlockBytes;
  h.n = n;
  h.blocks = (uint32_t)((n + kAnsBlockBytes - 1) / kAnsBlockBytes);
  make_freq(count, 2 * n, h.freq);
  uint32_t cum[17];
  cum[0] = 0;
  for (int s = 0; s < 16; s++) cum[s + 1] = cum[s] + h.freq[s];

  out.assign(sizeof(Header) + 4 * ((size_t)h.blocks + 1), 0);
  memcpy(out.data(), &h, sizeof(Header));
  const size_t area = out.size();
  std::vector<uint32_t> offset(h.blocks + 1, 0);
  std::vector<uint16_t> words[32];
  for (uint32_t b = 0; b < h.blocks; b++) {
    const uint64_t b0 = (uint64_t)b * kAnsBlockBytes;
    const uint32_t m = (uint32_t)(n - b0 < kAnsBlockBytes ? n - b0 : kAnsBlockBytes);
    const uint32_t nsym = 2 * m;
    uint32_t state[32];
    uint16_t nwords[32];
    for (int l = 0; l < 32; l++) {
      words[l].clear();
      uint32_t x = kLow;
      // encode this lane's symbols in reverse; its words come out last-first
      const int cnt = nsym > (uint32_t)l ? (int)((nsym - l + 31) / 32) : 0;
      for (int i = cnt - 1; i >= 0; i--) {
        const uint32_t j = (uint32_t)i * 32 + l;
        const uint8_t byte = in[b0 + j / 2];
        const int s = (j & 1) ? (byte >> 4) : (byte & 15);
        const uint32_t f = h.freq[s];
        const uint32_t x_max = ((kLow >> kProbBits) << 16) * f;
        while (x >= x_max) {
          words[l].push_back((uint16_t)(x & 0xffff));
          x >>= 16;
        }
        x = ((x / f) << kProbBits) + (x % f) + cum[s];
      }
      state[l] = x;
      nwords[l] = (uint16_t)words[l].size();
    }
    offset[b] = (uint32_t)(out.size() - area);
    const size_t at = out.size();
    size_t tot = 0;
    for (int l = 0; l < 32; l++) tot += words[l].size();
    out.resize(at + 32 * 4 + 32 * 2 + align4(2 * tot), 0);
    memcpy(out.data() + at, state, 32 * 4);
    memcpy(out.data() + at + 128, nwords, 32 * 2);
    uint8_t* wp = out.data() + at + 192;
    for (int l = 0; l < 32; l++)  // the decoder reads each lane's words first-emitted-last
      for (size_t k = words[l].size(); k-- > 0;) {
        memcpy(wp, &words[l][k], 2);
        wp += 2;
      }
  }
  offset[h.blocks] = (uint32_t)(out.size() - area);
  memcpy(out.data() + sizeof(Header), offset.data(), 4 * offset.size());
  return 0;
}

// Decoding table, one word per slot of the 12-bit probability range: symbol s in bits 0-3, its frequency
// f_s in bits 4-16, its cumulative frequency c_s in bits 17-28, so that a decoding step reads shared memory
// once (slot -> s, f_s, c_s). Built by every thread of the CTA from the stream's header.
__device__ __forceinline__ void build_decode_table(const Header* h, uint32_t* tab, uint32_t* fq) {
  if (threadIdx.x < 16) fq[threadIdx.x] = h->freq[threadIdx.x];
  __syncthreads();
  uint32_t c = 0;
  for (int s = 0; s < 16; s++) {
    const uint32_t f = fq[s];
    for (uint32_t i = threadIdx.x; i < f; i += blockDim.x) tab[c + i] = (uint32_t)s | (f << 4) | (c << 17);
    c += f;
  }
  __syncthreads();
}

// One decoding step of a lane's state: the symbol, and the state updated (without renormalisation).
__device__ __forceinline__ uint32_t ans_step(uint32_t& x, const uint32_t* tab) {
  const uint32_t slot = x & (kProbScale - 1);
  const uint32_t e = tab[slot];
  x = ((e >> 4) & 0x1fffu) * (x >> kProbBits) + slot - (e >> 17);
  return e & 15u;
}

// One warp per block. The warp first copies its block's words into shared memory (coalesced), so the
// serial state updates never wait on a global load; a block whose words exceed the stage (possible only
// for a block far from the stream's own statistics) is read from global memory instead. Lane l decodes
// symbols l, l + 32, ... of the block; even lane l and lane l + 1 hold the two nibbles of one byte and the
// even lane stores it. Word reads are bounded by the lane's word count (an inconsistent stream sets
// COLI_E_FORMAT instead of reading past it).
constexpr int kAnsWarps = 8;               // warps (blocks in flight) per CTA
constexpr uint32_t kAnsStageWords = 3072;  // 16-bit words staged per warp (6 KB; an incompressible block needs ~2100)

__global__ void __launch_bounds__(kAnsWarps * 32) ans_decode_kernel(const uint8_t* __restrict__ blob,
                                                                    uint8_t* __restrict__ out, int* err) {
  __shared__ uint32_t tab[kProbScale];
  __shared__ uint32_t fq[16];
  extern __shared__ __align__(16) uint16_t stage_dyn[];  // kAnsWarps x kAnsStageWords words
  const Header* h = reinterpret_cast<const Header*>(blob);
  build_decode_table(h, tab, fq);
  const uint32_t* offset = reinterpret_cast<const uint32_t*>(blob + sizeof(Header));
  const uint8_t* area = blob + sizeof(Header) + 4 * ((size_t)h->blocks + 1);
  const int lane = threadIdx.x & 31;
  const uint32_t b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= h->blocks) return;  // uniform per warp
  const uint8_t* blk = area + offset[b];
  const uint64_t b0 = (uint64_t)b * kAnsBlockBytes;
  const uint32_t m = (uint32_t)(h->n - b0 < kAnsBlockBytes ? h->n - b0 : kAnsBlockBytes);
  const uint32_t nsym = 2 * m;
  uint32_t x = reinterpret_cast<const uint32_t*>(blk)[lane];
  const uint32_t nw = reinterpret_cast<const uint16_t*>(blk + 128)[lane];
  uint32_t start = nw;  // exclusive prefix of the lanes' word counts
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, start, o);
    if (lane >= o) start += v;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, start, 31);  // the block's words
  start -= nw;
  const uint16_t* gw = reinterpret_cast<const uint16_t*>(blk + 192);
  uint16_t* sw = stage_dyn + (size_t)(threadIdx.x >> 5) * kAnsStageWords;
  const bool staged = total <= kAnsStageWords;
  if (staged)
    for (uint32_t k = lane; k < total; k += 32) sw[k] = gw[k];
  __syncwarp();
  const uint16_t* wp = (staged ? sw : gw) + start;
  uint32_t wi = 0;
  bool bad = false;
  const int cnt = (int)((nsym + 31) / 32);  // rounds; a lane past the end decodes nothing
  for (int i = 0; i < cnt; i++) {
    const uint32_t j = (uint32_t)i * 32 + lane;
    uint32_t s = 0;
    if (j < nsym) {
      s = ans_step(x, tab);
      if (x < kLow) {
        if (wi < nw) x = (x << 16) | wp[wi];
        else bad = true;
        wi++;
      }
    }
    const uint32_t hi = __shfl_down_sync(0xffffffffu, s, 1);
    if (!(lane & 1) && j < nsym) out[b0 + j / 2] = (uint8_t)(s | (hi << 4));
  }
  if (wi != nw || x != kLow) bad = true;  // every word used and the state back at its start
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, COLI_E_FORMAT);
}

// ------------------------------------------------------------------------------------------------
// Fused block decode + GEMV (PR #651, comment "Fused decode/matvec feasibility result": each block is
// decoded into on-chip memory and its row partials are computed at once, so only small partial sums
// are written instead of the raw tensor). The stream holds an int4 tensor W [O x I] in the packed
// format of coli_expert_upload: O rows of P = I / 2 bytes. One warp per block, as in the decoder: lane l
// decodes nibbles l, l + 32, ... of the block; nibble j is byte g = b0 + j / 2 of the tensor, i.e. row
// g / P and column 2 (g mod P) + (j & 1). The lane adds (n - 8) x[column] (times the column's group scale
// when gs > 0) to a running sum for its current row and parks it in shared memory when its row changes
// (a lane's bytes advance 16 at a time, so it meets each row once). At the block's end every row the
// block touched gets the sum of the 32 lanes' sums, in lane order: one partial per (block, row). The
// reduce kernel adds a row's partials in block order, applies a per-row scale (gs = 0) and the residual.
// ------------------------------------------------------------------------------------------------

constexpr int kGemvWarps = 8;
constexpr int kGemvMaxRows = 34;  // rows one 4096-byte block can touch when a row holds >= 128 bytes

// Rows a 4096-byte block can touch when rows hold P bytes.
__host__ __device__ constexpr int gemv_rows(uint32_t P) { return (int)((kAnsBlockBytes + P - 1) / P) + 1; }

__global__ void __launch_bounds__(kGemvWarps * 32) ans_gemv_kernel(const uint8_t* __restrict__ blob,
                                                                   const float* __restrict__ scales, int I, int gs,
                                                                   int G, const void* __restrict__ x, int x_dtype,
                                                                   float* __restrict__ part, int* err) {
  // dynamic: the warps' word stages, their row sums [nr][32] (nr rows a block can touch), the I activations
  extern __shared__ __align__(16) uint8_t gemv_dyn[];
  const uint32_t P = (uint32_t)I / 2;
  const int nr = gemv_rows(P);
  uint16_t* stage_all = reinterpret_cast<uint16_t*>(gemv_dyn);
  float* rows_all = reinterpret_cast<float*>(gemv_dyn + (size_t)kGemvWarps * kAnsStageWords * sizeof(uint16_t));
  float* xs = rows_all + (size_t)kGemvWarps * nr * 32;
  __shared__ uint32_t tab[kProbScale];
  __shared__ uint32_t fq[16];
  const Header* h = reinterpret_cast<const Header*>(blob);
  for (int i = threadIdx.x; i < I; i += blockDim.x) xs[i] = load_act(x, x_dtype, i);
  build_decode_table(h, tab, fq);  // (its barriers also publish xs)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t b = blockIdx.x * kGemvWarps + warp;
  if (b >= h->blocks) return;  // uniform per warp
  const uint32_t* offset = reinterpret_cast<const uint32_t*>(blob + sizeof(Header));
  const uint8_t* blk = blob + sizeof(Header) + 4 * ((size_t)h->blocks + 1) + offset[b];
  const uint64_t b0 = (uint64_t)b * kAnsBlockBytes;
  const uint32_t m = (uint32_t)(h->n - b0 < kAnsBlockBytes ? h->n - b0 : kAnsBlockBytes);
  const uint32_t nsym = 2 * m;
  const uint32_t r_first = (uint32_t)(b0 / P);
  float* rowsum = rows_all + (size_t)warp * nr * 32;  // [row - r_first][lane]
  for (int k = 0; k < nr; k++) rowsum[k * 32 + lane] = 0.f;
  uint32_t x_state = reinterpret_cast<const uint32_t*>(blk)[lane];
  const uint32_t nw = reinterpret_cast<const uint16_t*>(blk + 128)[lane];
  uint32_t start = nw;  // exclusive prefix of the lanes' word counts
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, start, o);
    if (lane >= o) start += v;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, start, 31);  // the block's words
  start -= nw;
  // the block's words into shared memory first (coalesced), as in the decoder, so that the state chains
  // do not wait on global loads; an oversized block reads them from global memory
  const uint16_t* gw = reinterpret_cast<const uint16_t*>(blk + 192);
  const bool staged = total <= kAnsStageWords;
  uint16_t* sw = stage_all + (size_t)warp * kAnsStageWords;
  if (staged)
    for (uint32_t k = lane; k < total; k += 32) sw[k] = gw[k];
  __syncwarp();
  const uint16_t* wp = (staged ? sw : gw) + start;
  // this lane's first byte, its row and its offset in the row; then 16 bytes further each step
  const uint64_t g0 = b0 + (lane >> 1);
  uint32_t r = (uint32_t)(g0 / P), cb = (uint32_t)(g0 - (uint64_t)r * P);
  uint32_t cur = r;
  float acc = 0.f;
  uint32_t wi = 0;
  bool bad = false;
  const int cnt = (int)((nsym + 31) / 32);
  for (int i = 0; i < cnt; i++) {
    const uint32_t j = (uint32_t)i * 32 + lane;
    if (j < nsym) {
      // the activation (and group scale) of this nibble's column first: they do not depend on the state
      const uint32_t col = 2 * cb + (lane & 1);
      const float xv = xs[col];
      const float sv = gs > 0 ? __ldg(scales + (size_t)r * G + col / (uint32_t)gs) : 1.f;
      const uint32_t s = ans_step(x_state, tab);
      if (x_state < kLow) {
        if (wi < nw) x_state = (x_state << 16) | wp[wi];
        else bad = true;
        wi++;
      }
      if (r != cur) {  // the lane has left row `cur` for good
        rowsum[(cur - r_first) * 32 + lane] = acc;
        acc = 0.f;
        cur = r;
      }
      float t = (float)((int)s - 8) * xv;
      if (gs > 0) t *= sv;
      acc += t;
      cb += 16;
      if (cb >= P) {
        cb -= P;
        r++;
      }
    }
  }
  rowsum[(cur - r_first) * 32 + lane] = acc;
  __syncwarp();
  const uint32_t r_last = (uint32_t)((b0 + m - 1) / P);
  for (uint32_t k = lane; k <= r_last - r_first; k += 32) {
    float t = 0.f;
    for (int l = 0; l < 32; l++) t += rowsum[k * 32 + l];
    part[(size_t)b * kGemvMaxRows + k] = t;
  }
  if (wi != nw || x_state != kLow) bad = true;  // every word used and the state back at its start
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, COLI_E_FORMAT);
}

// y[r] = resid[r] + (s_r for gs = 0) * (the partials of the blocks touching row r, in block order).
__global__ void ans_gemv_reduce_kernel(const float* __restrict__ part, int O, int I, int gs,
                                       const float* __restrict__ scales, const void* resid, int dtype, void* y) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= O) return;
  const uint64_t P = (uint64_t)I / 2;
  const uint64_t g_lo = (uint64_t)r * P, g_hi = g_lo + P - 1;
  float t = 0.f;
  for (uint64_t b = g_lo / kAnsBlockBytes; b <= g_hi / kAnsBlockBytes; b++) {
    const uint64_t r_first = b * kAnsBlockBytes / P;
    t += part[b * kGemvMaxRows + (r - r_first)];
  }
  if (gs == 0) t *= __ldg(scales + r);
  if (resid) t = load_act(resid, dtype, r) + t;
  if (dtype == COLI_DTYPE_F32)
    static_cast<float*>(y)[r] = t;
  else
    static_cast<uint16_t*>(y)[r] = f32_to_bf16_rn(t);
}

int launch_ans_gemv(coli_ctx* ctx, const AnsStream& st, const float* scales, int O, int I, int gs, const void* x,
                    int x_dtype, const void* resid, void* y) {
  const size_t pbytes = (size_t)st.blocks * kGemvMaxRows * sizeof(float);
  int rc = ensure_workspace(ctx, pbytes);
  if (rc != COLI_OK) return rc;
  float* part = reinterpret_cast<float*>(ctx->ws.base);
  const size_t smem = (size_t)kGemvWarps * kAnsStageWords * sizeof(uint16_t) +
                      (size_t)kGemvWarps * gemv_rows((uint32_t)I / 2) * 32 * sizeof(float) + (size_t)I * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(ans_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "ans_w4_linear: shared memory attribute");
  const int G = gs > 0 ? (I + gs - 1) / gs : 1;
  {
    ProfScope prof(ctx, COLI_KERNEL_LINEAR);
    ans_gemv_kernel<<<(st.blocks + kGemvWarps - 1) / kGemvWarps, kGemvWarps * 32, smem, ctx->stream>>>(
        st.d_blob, scales, I, gs, G, x, x_dtype, part, ctx->d_status);
    ans_gemv_reduce_kernel<<<(O + 255) / 256, 256, 0, ctx->stream>>>(part, O, I, gs, scales, resid, x_dtype, y);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "ans_w4_linear launch");
  return COLI_OK;
}

int ans_blocks(const void* blob_host) { return (int)reinterpret_cast<const Header*>(blob_host)->blocks; }

namespace {
std::mutex g_streams_mu;
std::map<coli_ctx*, std::vector<AnsStream>> g_streams;  // handle = index + 1
}  // namespace

std::vector<AnsStream>& ans_streams(coli_ctx* ctx) {
  std::lock_guard<std::mutex> lock(g_streams_mu);
  return g_streams[ctx];
}

void ans_release_all(coli_ctx* ctx) {
  std::lock_guard<std::mutex> lock(g_streams_mu);
  auto it = g_streams.find(ctx);
  if (it == g_streams.end()) return;
  for (auto& s : it->second)
    if (s.d_blob) cudaFree(s.d_blob);
  g_streams.erase(it);
}

int launch_ans_decode(coli_ctx* ctx, const uint8_t* blob, int blocks, uint8_t* out) {
  const size_t smem = (size_t)kAnsWarps * kAnsStageWords * sizeof(uint16_t);
  cudaError_t e0 = cudaFuncSetAttribute(ans_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e0 != cudaSuccess) return cuda_fail(ctx, e0, "ans_decode: shared memory attribute");
  ans_decode_kernel<<<(blocks + kAnsWarps - 1) / kAnsWarps, kAnsWarps * 32, smem, ctx->stream>>>(blob, out,
                                                                                               ctx->d_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "ans_decode launch");
  return COLI_OK;
}

}  // namespace coli
