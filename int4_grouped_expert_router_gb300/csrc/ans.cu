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

// One warp per block. The warp first copies its block's words into shared memory (coalesced), so the
// serial state updates never wait on a global load; a block whose words exceed the stage (possible only
// for a block far from the stream's own statistics) is read from global memory instead. Lane l decodes
// symbols l, l + 32, ... of the block; even lane l and lane l + 1 hold the two nibbles of one byte and the
// even lane stores it. Word reads are bounded by the lane's word count (an inconsistent stream sets
// COLI_E_FORMAT instead of reading past it).
constexpr int kAnsWarps = 4;               // warps (blocks in flight) per CTA
constexpr uint32_t kAnsStageWords = 4096;  // 16-bit words staged per warp (8 KB)

__global__ void __launch_bounds__(kAnsWarps * 32) ans_decode_kernel(const uint8_t* __restrict__ blob,
                                                                    uint8_t* __restrict__ out, int* err) {
  __shared__ uint8_t sym_of[kProbScale];
  __shared__ uint16_t stage[kAnsWarps][kAnsStageWords];
  __shared__ uint32_t fq[16], cm[16];
  const Header* h = reinterpret_cast<const Header*>(blob);
  if (threadIdx.x < 16) fq[threadIdx.x] = h->freq[threadIdx.x];
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t c = 0;
    for (int s = 0; s < 16; s++) {
      cm[s] = c;
      c += fq[s];
    }
  }
  __syncthreads();
  for (int s = 0; s < 16; s++)
    for (uint32_t i = threadIdx.x; i < fq[s]; i += blockDim.x) sym_of[cm[s] + i] = (uint8_t)s;
  __syncthreads();
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
  uint16_t* sw = stage[threadIdx.x >> 5];
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
      const uint32_t slot = x & (kProbScale - 1);
      s = sym_of[slot];
      x = fq[s] * (x >> kProbBits) + slot - cm[s];
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
  ans_decode_kernel<<<(blocks + kAnsWarps - 1) / kAnsWarps, kAnsWarps * 32, 0, ctx->stream>>>(blob, out,
                                                                                            ctx->d_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "ans_decode launch");
  return COLI_OK;
}

}  // namespace coli
