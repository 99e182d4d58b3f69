// warp_rows_kernel.cuh — multi-row path: one warp selects one row, a CTA holds
// kWrWarps rows at a time, and a persistent grid walks the batch.
//
// For many short rows (the decode-shaped indexer call: thousands of rows of a
// few ten thousand elements) a whole CTA per row spends most of its time in
// CTA-wide barriers between short phases. Here every row is owned by a single
// warp, so all coordination is warp-synchronous (ballots, shuffles,
// __syncwarp) and the SM keeps dozens of independent rows in flight, which is
// what hides HBM latency. Per row:
//
//  T  threshold t (an order key): the warp's previous row's k-th key lowered by
//     a margin, or, for a warp's first row, a value read off a sample of vector
//     maxima (16 evenly spaced blocks of 32 vectors), or of the elements of
//     those vectors when k is over a quarter of the row's vectors. t is only a
//     guess; the step below checks it.
//  S  stream the row once through a per-warp shared-memory ring of 2 KB bulk
//     async copies. In each chunk lane j owns 4 consecutive 16-byte vectors
//     (64 contiguous bytes); it marks its elements >= t (or NaN) in one 32-bit
//     mask with packed compares, one warp prefix sum over the lanes' counts
//     places the chunk's candidates, and each lane copies its marked elements
//     (read back from the chunk in shared memory) into the warp's candidate
//     buffer. Lanes own consecutive vectors, so candidates land in index order.
//     The guess holds iff k <= candidates <= capacity (and no NaN): then the
//     candidates contain the row's top k.
//  R  exact k-th key K* among the candidates: 256-bin histogram levels, the
//     first over the 256 top-16-bit keys from t up (it also spots a NaN),
//     each further level narrowing the range by 8 bits.
//  C  output: keep key > K*, and the first keys == K* in index order until k
//     are taken. For sorted_index 1, one ordered pass writes them in ascending
//     index order (at no extra cost); otherwise the keys above K* go first
//     (one ballot per 32 candidates) and a short pass adds the ties.
//
// A row whose guess fails is retried (sample threshold, a sample rank adapted to
// the count seen, the exact k-th vector maximum, or for dense rows the exact top
// 16 key bits of the k-th element) with direct passes over the
// row; a row that still fails (massive ties, a NaN, k above the number of
// finite vectors) takes the exact fallback: 8-bit radix levels over every
// element of the row, then one ordered output pass. Rows with a NaN set the
// device flag there.
//
// Sources: deepseek.csdn.net, "DeepSeek 一次开源三个仓库", section 三 (算子层):
// the threshold filter into a candidate buffer and its compaction to K;
// deepseek-v4-pro.uk (zh-tw), "深入 DeepSeek V4.1 全新開放推論工具包", section
// "DeepSelect：快速且刻意狹義的 TopK": bf16 and fp32, k <= 4096, the always-on
// NaN check; github-research.aiutil.com, "deepseek-ai/DeepSelect", section
// 关键技术亮点: batch sizes from 1 upwards and effective memory bandwidth as the
// metric (every row is read from HBM once on the common path).
#pragma once

#include "topk_kernel.cuh"

namespace ds_topk_dev {

constexpr int kWrWarps = 8;                // rows in flight per CTA
constexpr int kWrThreads = 32 * kWrWarps;
constexpr int kWrMaxLen = 65536;           // candidate indices are kept in 16 bits
constexpr int kWrMaxK = 1024;
constexpr int kWrSampleBlocks = 16;        // first-row sample: 16 blocks of 32 vectors
constexpr int kWrChunk = 2048;             // bytes per bulk copy of a row (128 vectors)
constexpr int kWrChunkVecs = kWrChunk / 16;
constexpr int kWrLaneVecs = kWrChunkVecs / 32;  // consecutive vectors a lane owns per chunk
constexpr int kWrMaxDepth = 3;             // chunks in flight per warp
// Bounded mbarrier polls (a test build sets a short limit to make a wait run out).
#ifndef DS_TOPK_WAIT_LIMIT
#define DS_TOPK_WAIT_LIMIT (1u << 22)
#endif
constexpr uint32_t kWrWaitLimit = DS_TOPK_WAIT_LIMIT;
constexpr uint32_t kWrSuspendNs = 1000;      // a poll may sleep this long before it fails
constexpr int kSelU = 4;                     // candidates per lane in flight in the selection passes

static_assert(kWrLaneVecs == 4, "a lane's candidate mask holds 4 vectors of 8 bf16 elements");

struct WrParams {
  const char* x;
  int64_t batch;
  int64_t row_stride_bytes;
  int32_t len;
  int32_t cap;            // candidate slots per warp (multiple of 32)
  int32_t depth;          // chunks of the streaming ring (2 or 3)
  int32_t k;
  int32_t return_value;
  int32_t ordered;        // outputs in ascending index order (sorted_index 1)
  void* out_values;
  void* out_indices;      // int32 or int64 (idx64)
  int32_t idx64;
  int32_t* flag;
};

// Per-warp shared memory: streaming ring (depth x 2 KB) | 256-bin histogram |
// mbarriers | candidate words | candidate indices (fp32 only). bf16 candidate
// word: input bits | index << 16; fp32: input bits, index apart.
constexpr int kWrFixedBytes = kRadix * 4 + kWrMaxDepth * 8 + 8;
__host__ __device__ constexpr int64_t wr_warp_bytes(int es, int64_t cap, int depth) {
  return depth * kWrChunk + kWrFixedBytes + cap * 4 + (es == 4 ? cap * 2 : 0);
}

template <int ES>
__device__ __forceinline__ uint32_t wr_key_floor() {
  return ES == 2 ? 0x0080u : 0x00800000u;  // key(-inf)
}

// NaN-propagating maximum of a vector, packed (bf16x2 or one f32).
template <int ES>
__device__ __forceinline__ uint32_t vec_max(const uint4& w) {
  if constexpr (ES == 2) {
    return bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w));
  } else {
    return f32_max_nan(f32_max_nan(w.x, w.y), f32_max_nan(w.z, w.w));
  }
}

// ---- bulk copies into shared memory, completed through an mbarrier ----------------
__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void mbar_init(uint64_t* m, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(m)), "r"(count) : "memory");
}
// One arrival that also announces `bytes` of incoming copies, then the copy of
// `bytes` (a multiple of 16, both addresses 16-byte aligned) that completes them.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* m) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(m)), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(m))
      : "memory");
}
// Polls the mbarrier phase with the given parity at most kWrWaitLimit times.
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity) {
  const uint32_t a = smem_addr(m);
  for (uint32_t i = 0; i < kWrWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(a), "r"(parity), "r"(kWrSuspendNs) : "memory");
    if (ok) return true;
  }
  return false;
}

// Bins [8*lane, 8*lane+8) of a 256-bin histogram; returns the bin b with
//   sum(h[> b]) < need <= sum(h[>= b])
// (the bin of the need-th largest key) and sum(h[> b]) in *above. The caller
// guarantees sum(h) >= need. Warp-synchronous.
__device__ __forceinline__ uint32_t wr_find_bin(const uint32_t* h, uint32_t need, uint32_t* above,
                                                uint32_t* count) {
  const int lane = threadIdx.x & 31;
  const uint4 c0 = reinterpret_cast<const uint4*>(h)[lane * 2];
  const uint4 c1 = reinterpret_cast<const uint4*>(h)[lane * 2 + 1];
  const uint32_t c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += c[j];
  uint32_t suf = s;  // sum over lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, suf, o);
    if (lane + o < 32) suf += t;
  }
  const uint32_t above_lane = suf - s;
  const bool mine = above_lane < need && need <= suf;
  uint32_t bin = 0, ab = 0, cnt = 0;
  if (mine) {
    uint32_t run = above_lane;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (run + c[j] >= need) {
        bin = static_cast<uint32_t>(lane * 8 + j);
        ab = run;
        cnt = c[j];
        break;
      }
      run += c[j];
    }
  }
  const uint32_t who = __ballot_sync(0xFFFFFFFFu, mine);
  const int src = who ? __ffs(who) - 1 : 0;
  *above = __shfl_sync(0xFFFFFFFFu, ab, src);
  *count = __shfl_sync(0xFFFFFFFFu, cnt, src);
  return __shfl_sync(0xFFFFFFFFu, bin, src);
}

__device__ __forceinline__ void wr_clear_hist(uint32_t* h) {
  const int lane = threadIdx.x & 31;
  reinterpret_cast<uint4*>(h)[lane * 2] = make_uint4(0, 0, 0, 0);
  reinterpret_cast<uint4*>(h)[lane * 2 + 1] = make_uint4(0, 0, 0, 0);
  __syncwarp();
}

// Candidate bits of one 16-byte vector against threshold value tval (tv2: its
// bf16 bits in both halves): bit e set iff element e is not below the threshold
// or is NaN (unordered compares), so every NaN becomes a candidate and is seen
// by the selection. bf16: 8 bits from 4 packed compares (setp.geu.bf16x2 sets
// the first predicate from the low half, i.e. the even element); fp32: 4 bits.
template <int ES>
__device__ __forceinline__ uint32_t vec_cand_bits(const uint4& w, float tval, uint32_t tv2) {
  uint32_t m;
  if constexpr (ES == 2) {
    (void)tval;
    asm("{\n\t.reg .pred a0, a1, b0, b1, c0, c1, d0, d1;\n\t"
        "setp.geu.bf16x2 a0|a1, %1, %5;\n\t"
        "setp.geu.bf16x2 b0|b1, %2, %5;\n\t"
        "setp.geu.bf16x2 c0|c1, %3, %5;\n\t"
        "setp.geu.bf16x2 d0|d1, %4, %5;\n\t"
        "selp.u32 %0, 1, 0, a0;\n\t"
        "@a1 or.b32 %0, %0, 2;\n\t"
        "@b0 or.b32 %0, %0, 4;\n\t"
        "@b1 or.b32 %0, %0, 8;\n\t"
        "@c0 or.b32 %0, %0, 16;\n\t"
        "@c1 or.b32 %0, %0, 32;\n\t"
        "@d0 or.b32 %0, %0, 64;\n\t"
        "@d1 or.b32 %0, %0, 128;\n\t}"
        : "=r"(m) : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(tv2));
  } else {
    (void)tv2;
    m = static_cast<uint32_t>(!(__uint_as_float(w.x) < tval)) |
        static_cast<uint32_t>(!(__uint_as_float(w.y) < tval)) << 1 |
        static_cast<uint32_t>(!(__uint_as_float(w.z) < tval)) << 2 |
        static_cast<uint32_t>(!(__uint_as_float(w.w) < tval)) << 3;
  }
  return m;
}

template <int ES>
struct WarpRow {
  using T = Traits<ES>;
  static constexpr int VEC = T::kVec;
  static constexpr int KB = T::kKeyBits;
  static constexpr uint32_t kFull = 0xFFFFFFFFu;

  const WrParams& p;
  uint4* chunks;  // streaming ring, depth x kWrChunkVecs vectors
  uint32_t* hist;
  uint64_t* mbar;
  uint32_t* cw;   // candidate words
  uint16_t* ci;   // candidate indices (fp32)
  int lane;
  uint32_t lt;
  int rot;        // rotation of the lane's four loads (conflict-free shared-memory reads)

  __device__ WarpRow(const WrParams& prm, unsigned char* base)
      : p(prm),
        chunks(reinterpret_cast<uint4*>(base)),
        hist(reinterpret_cast<uint32_t*>(base + prm.depth * kWrChunk)),
        mbar(reinterpret_cast<uint64_t*>(base + prm.depth * kWrChunk + kRadix * 4)),
        cw(reinterpret_cast<uint32_t*>(base + prm.depth * kWrChunk + kWrFixedBytes)),
        ci(reinterpret_cast<uint16_t*>(base + prm.depth * kWrChunk + kWrFixedBytes) + 2 * prm.cap),
        lane(threadIdx.x & 31),
        lt(lanemask_lt()),
        rot((threadIdx.x >> 1) & 3) {}

  // ---- where a row lies: the 16-byte blocks that overlap it ---------------------
  // A row may start anywhere on its element size. It is read as the 16-byte
  // aligned blocks that overlap [0, len): block v holds row elements
  // v*VEC + e - lead for e = 0..VEC-1. Elements outside [0, len) that share a
  // block with row elements are masked before anything looks at them; no block
  // without a row element is read (and an aligned 16-byte block never crosses a
  // page, so the reads stay inside the row's pages).
  struct Geo {
    const char* base;  // the first block
    int lead;          // elements of the first block before the row's element 0
    int nv;            // blocks overlapping the row
    int nch;           // bulk chunks covering them
  };
  __device__ __forceinline__ Geo geo(int64_t row) const {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.x + row * p.row_stride_bytes);
    Geo g;
    g.base = reinterpret_cast<const char*>(a & ~static_cast<uintptr_t>(15));
    g.lead = static_cast<int>((a & 15u) / ES);
    g.nv = (g.lead + p.len + VEC - 1) / VEC;
    g.nch = (g.nv + kWrChunkVecs - 1) / kWrChunkVecs;
    return g;
  }
  // Block v with every element outside the row set to -inf (only the first and
  // the last block can hold such elements).
  __device__ __forceinline__ uint4 load(const Geo& g, int v) const {
    uint4 w = ld_nc_v4(g.base + static_cast<int64_t>(v) * 16);
    if (v == 0 || v == g.nv - 1) {
      uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const int idx = v * VEC + e - g.lead;
        if (idx < 0 || idx >= p.len) {
          if constexpr (ES == 2) {
            const int sh = (e & 1) * 16;
            ws[e >> 1] = (ws[e >> 1] & ~(0xFFFFu << sh)) | (0xFF80u << sh);
          } else {
            ws[e] = 0xFF800000u;
          }
        }
      }
      w = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    }
    return w;
  }
  // Mask of the row elements among a lane's 4 blocks v0 .. v0+3 (bit VEC*u + e
  // for element e of block v0 + u).
  __device__ __forceinline__ uint32_t valid_bits(const Geo& g, int v0) const {
    constexpr int W = kWrLaneVecs * VEC;
    const int lo = g.lead - v0 * VEC;  // bit of row element 0
    const int a = lo > 0 ? lo : 0;
    const int b = lo + p.len < W ? lo + p.len : W;
    if (b <= a) return 0u;
    const uint32_t upto = b >= 32 ? 0xFFFFFFFFu : ((1u << b) - 1u);
    return upto & ~((1u << a) - 1u);
  }

  // Top 16 bits of the key of a packed maximum (bf16: the key itself).
  __device__ __forceinline__ uint32_t key16(uint32_t vmax) const {
    const uint32_t k = key_of<ES>(finish_max<ES>(vmax));
    return ES == 2 ? k : (k >> 16);
  }

  // ---- T: first-row threshold from a sample of vector maxima ----------------------
  // Rows of at most 512 vectors are read whole, and the threshold is exact: the
  // k-th largest vector maximum, which at least k elements reach. Longer rows
  // are sampled in 16 evenly spaced blocks of 32 consecutive vectors (coalesced,
  // 1/8 of a 64 KB row's cache lines, which the stream then finds in L2), and the
  // threshold is the q-th largest sampled maximum, q about 1.2 k times the
  // sampled fraction plus a margin: a guess that the stream verifies. Dense rows
  // rank the sampled elements with the same q (the sampled fraction is the same).
  __device__ __forceinline__ int sample_size(const Geo& g) const {
    return g.nv <= 32 * kWrSampleBlocks ? g.nv : 32 * kWrSampleBlocks;
  }
  // The rank q of the sampled maximum used as the first-row threshold.
  __device__ __forceinline__ uint32_t default_rank(const Geo& g) const {
    if (g.nv <= 32 * kWrSampleBlocks) return static_cast<uint32_t>(p.k);
    return static_cast<uint32_t>((static_cast<int64_t>(6 * p.k) * sample_size(g) / 5 + g.nv - 1) / g.nv + 8);
  }
  // A rank for a second try after the threshold of rank q gave n candidates:
  // candidates grow about in proportion to q.
  __device__ __forceinline__ uint32_t adapted_rank(uint32_t q, int n) const {
    uint32_t r;
    if (n > p.cap) r = static_cast<uint32_t>(static_cast<int64_t>(q) * (3 * p.cap / 4) / n);
    else r = static_cast<uint32_t>(static_cast<int64_t>(q) * (5 * p.k / 4) / (n > 0 ? n : 1)) + 4;
    return r < 1u ? 1u : r;
  }
  // Dense rows, where k is over a quarter of the row's vectors, rank element keys
  // instead: with several selected elements per vector, the count of elements
  // above the q-th largest vector maximum is no longer close to q.
  __device__ __forceinline__ bool dense(const Geo& g) const { return 4 * p.k > g.nv; }

  // The q-th largest top-16 key bits among the elements of the vectors
  // i * vstride + lane (i < steps, vectors past the row skipped): two 8-bit
  // histogram levels, each over the vectors read again (from L1 or L2).
  __device__ uint32_t elem_threshold(const Geo& g, uint32_t q, int steps, int vstride) const {
    uint32_t b1 = 0, need = q;
    for (int level = 0; level < 2; ++level) {
      wr_clear_hist(hist);
      for (int i = 0; i < steps; ++i) {
        const int v = i * vstride + lane;
        if (v >= g.nv) continue;
        const uint4 w = load(g, v);  // elements outside the row read as -inf
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const uint32_t kk = key_of<ES>(elem_bits<ES>(w, e)) >> (KB - 16);
          if (level == 0) atomicAdd(&hist[kk >> 8], 1u);
          else if ((kk >> 8) == b1) atomicAdd(&hist[kk & 0xFFu], 1u);
        }
      }
      __syncwarp();
      uint32_t above, cnt;
      const uint32_t b = wr_find_bin(hist, need, &above, &cnt);
      __syncwarp();
      need -= above;
      b1 = level == 0 ? b : ((b1 << 8) | b);
    }
    uint32_t t = b1;
    if constexpr (ES == 4) t <<= 16;
    return t < wr_key_floor<ES>() ? wr_key_floor<ES>() : t;
  }

  __device__ uint32_t sample_threshold(const Geo& g, uint32_t q) const {
    const int nvec = g.nv;
    constexpr int kPer = kWrSampleBlocks;  // vectors per lane
    const bool whole = nvec <= 32 * kPer;
    const int ns = whole ? nvec : 32 * kPer;
    const int bstride = whole ? 32 : (nvec - 32) / (kPer - 1);  // block starts: i * bstride
    if (dense(g)) {  // q ranks the sampled elements, VEC per sampled vector
      if (q > static_cast<uint32_t>(ns * VEC)) return wr_key_floor<ES>();
      return elem_threshold(g, q, kPer, bstride);
    }
    if (q > static_cast<uint32_t>(ns)) return wr_key_floor<ES>();
    uint32_t kk[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int v = i * bstride + lane;
      kk[i] = (whole ? v < nvec : true) ? key16(vec_max<ES>(load(g, v))) : 0xFFFFFFFFu;
    }
    wr_clear_hist(hist);
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (kk[i] != 0xFFFFFFFFu) atomicAdd(&hist[kk[i] >> 8], 1u);
    __syncwarp();
    uint32_t above, cnt;
    const uint32_t b1 = wr_find_bin(hist, q, &above, &cnt);
    __syncwarp();
    wr_clear_hist(hist);
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (kk[i] != 0xFFFFFFFFu && (kk[i] >> 8) == b1) atomicAdd(&hist[kk[i] & 0xFFu], 1u);
    __syncwarp();
    const uint32_t b2 = wr_find_bin(hist, q - above, &above, &cnt);
    __syncwarp();
    uint32_t t = (b1 << 8) | b2;
    if constexpr (ES == 4) t <<= 16;
    return t < wr_key_floor<ES>() ? wr_key_floor<ES>() : t;
  }

  __device__ __forceinline__ void put(int pos, uint32_t bits, int idx) const {
    if constexpr (ES == 2) {
      cw[pos] = bits | (static_cast<uint32_t>(idx) << 16);
    } else {
      cw[pos] = bits;
      ci[pos] = static_cast<uint16_t>(idx);
    }
  }
  __device__ __forceinline__ uint32_t bits_at(int pos) const {
    return ES == 2 ? (cw[pos] & 0xFFFFu) : cw[pos];
  }
  __device__ __forceinline__ int idx_at(int pos) const {
    return ES == 2 ? static_cast<int>(cw[pos] >> 16) : static_cast<int>(ci[pos]);
  }

  // ---- S: candidates of a group of 32 x 4 consecutive vectors ---------------------
  // M: the lane's candidate mask over its 4 consecutive vectors (bit VEC*v + e:
  // element e of the lane's vector v); ibase: the row index of the lane's first
  // element. The lanes' candidates are appended at *ccount (warp-uniform) in
  // index order (writes stop at cap; the count does not). bits_of(b) returns
  // the element bits behind mask bit b.
  template <typename BitsOf>
  __device__ __forceinline__ void emit(uint32_t M, int ibase, int* ccount, BitsOf bits_of) const {
    if (__ballot_sync(kFull, M != 0u) == 0u) return;  // warp-uniform: nothing here
    const uint32_t cnt = __popc(M);
    const uint32_t excl = warp_excl_scan(cnt);
    const int tot = static_cast<int>(__shfl_sync(kFull, excl + cnt, 31));
    int pos = *ccount + static_cast<int>(excl);
    while (M) {
      const int b = __ffs(M) - 1;
      M &= M - 1;
      if (pos < p.cap) put(pos, bits_of(b), ibase + b);
      ++pos;
    }
    *ccount += tot;
  }

  // Candidate mask of the lane's 4 consecutive vectors held in r[0..3], where
  // r[u] is the lane's vector vu(u) (0..3) and only vectors below `valid` count.
  __device__ __forceinline__ uint32_t lane_mask(const uint4 (&r)[kWrLaneVecs], const int (&vu)[kWrLaneVecs],
                                                int valid, float tval, uint32_t tv2) const {
    uint32_t M = 0;
#pragma unroll
    for (int u = 0; u < kWrLaneVecs; ++u) {
      const uint32_t b = vec_cand_bits<ES>(r[u], tval, tv2);
      M |= (vu[u] < valid ? b : 0u) << (VEC * vu[u]);
    }
    return M;
  }

  // Element bits behind mask bit b of the lane's 4 vectors, from registers (the
  // retry passes, which read the row straight from global memory).
  __device__ __forceinline__ static uint32_t reg_bits(const uint4 (&r)[kWrLaneVecs], int b) {
    const int v = b / VEC, e = b % VEC;
    const uint4 a = (v & 2) ? ((v & 1) ? r[3] : r[2]) : ((v & 1) ? r[1] : r[0]);
    return elem_bits<ES>(a, e);
  }

  // The retry pass: the row straight from global memory (it was just streamed,
  // so mostly from L2), 4 consecutive blocks per lane. Returns the candidate
  // count (it may exceed cap; writes stop there).
  __device__ int direct_pass(const Geo& g, uint32_t tk) const {
    const float tval = key_threshold_value<ES>(tk);
    const uint32_t tv2 = (__float_as_uint(tval) >> 16) * 0x00010001u;
    const int vu[kWrLaneVecs] = {0, 1, 2, 3};
    int ccount = 0;
    for (int c0 = 0; c0 < g.nv; c0 += kWrChunkVecs) {
      const int v0 = c0 + lane * kWrLaneVecs;
      uint4 r[kWrLaneVecs];
#pragma unroll
      for (int u = 0; u < kWrLaneVecs; ++u)
        r[u] = v0 + u < g.nv ? ld_nc_v4(g.base + static_cast<int64_t>(v0 + u) * 16) : make_uint4(0, 0, 0, 0);
      uint32_t M = lane_mask(r, vu, g.nv - v0, tval, tv2);
      if (c0 == 0 || c0 + kWrChunkVecs >= g.nv) M &= valid_bits(g, v0);  // warp-uniform
      emit(M, v0 * VEC - g.lead, &ccount, [&](int b) { return reg_bits(r, b); });
    }
    return ccount;
  }

  // ---- the streaming ring: chunks of the warp's rows, in order, depth ahead -------
  struct Stream {
    const char* src;    // source of the next chunk to copy (null: none left)
    int64_t prow;       // its row
    int pleft;          // chunks of that row still to copy, src's included
    uint32_t plast;     // bytes of that row's last chunk
    int pslot;          // ring slot it goes to
    int cslot;          // ring slot of the next chunk to read
    uint32_t cphase;    // mbarrier phase parity that chunk completes
    uint32_t issued;    // chunks copied so far
    uint32_t consumed;  // chunks read so far
  };
  // Points the producer at row `row` (or at nothing past the batch).
  __device__ __forceinline__ void stream_row(Stream& st, int64_t row) const {
    st.prow = row;
    if (row < p.batch) {
      const Geo g = geo(row);
      st.src = g.base;
      st.pleft = g.nch;
      st.plast = static_cast<uint32_t>(g.nv - (g.nch - 1) * kWrChunkVecs) * 16u;
    } else {
      st.src = nullptr;
    }
  }
  __device__ __forceinline__ void stream_begin(Stream& st, int64_t first) const {
    stream_row(st, first);
    st.pslot = st.cslot = 0;
    st.cphase = st.issued = st.consumed = 0u;
  }
  // Copies the next chunk of the warp's row sequence into the ring, if any.
  __device__ __forceinline__ void produce_one(Stream& st, int64_t row_step) const {
    if (st.src == nullptr) return;
    const uint32_t bytes = st.pleft == 1 ? st.plast : static_cast<uint32_t>(kWrChunk);
    if (lane == 0) bulk_load(chunks + st.pslot * kWrChunkVecs, st.src, bytes, mbar + st.pslot);
    if (++st.pslot == p.depth) st.pslot = 0;
    ++st.issued;
    if (--st.pleft == 0) {
      stream_row(st, st.prow + row_step);
    } else {
      st.src += kWrChunk;
    }
  }
  // The candidate pass over one row, fed by the ring: a chunk's slot is refilled
  // with the chunk `depth` places further on once its candidates are copied out.
  // Returns false if a copy never completed within the poll limit (the warp must
  // then stop); else the candidate count in *n (it may exceed cap).
  __device__ bool stream_pass(Stream& st, int64_t row_step, const Geo& g, uint32_t tk, int* n) const {
    const float tval = key_threshold_value<ES>(tk);
    const uint32_t tv2 = (__float_as_uint(tval) >> 16) * 0x00010001u;
    int vu[kWrLaneVecs];
#pragma unroll
    for (int u = 0; u < kWrLaneVecs; ++u) vu[u] = (u + rot) & (kWrLaneVecs - 1);
    int ccount = 0;
    for (int c = 0; c < g.nch; ++c) {
      const int slot = st.cslot;
      if (!__all_sync(kFull, mbar_wait(mbar + slot, st.cphase))) return false;
      if (++st.cslot == p.depth) {
        st.cslot = 0;
        st.cphase ^= 1u;
      }
      // the lane's 64 bytes; load u reads block vu[u], so the 8 lanes of each
      // quarter-warp touch 8 distinct 16-byte bank groups
      const uint4* lv = chunks + slot * kWrChunkVecs + lane * kWrLaneVecs;
      const int v0 = c * kWrChunkVecs + lane * kWrLaneVecs;
      uint4 r[kWrLaneVecs];
#pragma unroll
      for (int u = 0; u < kWrLaneVecs; ++u) r[u] = lv[vu[u]];
      uint32_t M = lane_mask(r, vu, kWrLaneVecs, tval, tv2);
      // the first and the last chunk hold elements outside the row (and stale
      // blocks past the row's last one): only row elements count
      if (c == 0 || c == g.nch - 1) M &= valid_bits(g, v0);  // warp-uniform
      const char* lb = reinterpret_cast<const char*>(lv);
      emit(M, v0 * VEC - g.lead, &ccount, [&](int b) {
        return ES == 2 ? static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(lb)[b])
                       : reinterpret_cast<const uint32_t*>(lb)[b];
      });
      __syncwarp();  // every lane is done with the slot: refill it
      ++st.consumed;
      produce_one(st, row_step);
    }
    *n = ccount;
    return true;
  }
  // Waits (bounded) for every copy still in flight.
  __device__ void drain(Stream& st) const {
    while (st.consumed != st.issued) {
      mbar_wait(mbar + st.cslot, st.cphase);
      if (++st.cslot == p.depth) {
        st.cslot = 0;
        st.cphase ^= 1u;
      }
      ++st.consumed;
    }
  }

  // ---- C: the output pass ----------------------------------------------------------
  // Every candidate with key > kth, and the first `need` with key == kth in index
  // order. Ordered output: one pass, positions in ascending index order. Any
  // other order: the keys above kth with one ballot per 32 candidates, then the
  // ties in a short pass that stops once `need` of them are written.
  template <bool IDX64, bool RETV>
  __device__ __forceinline__ void write_out(int64_t row, int n, uint32_t kth, uint32_t need) const {
    using VT = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
    const int64_t obase = row * p.k;
    int32_t* oi32 = static_cast<int32_t*>(p.out_indices) + obase;
    int64_t* oi64 = static_cast<int64_t*>(p.out_indices) + obase;
    VT* ov = RETV ? static_cast<VT*>(p.out_values) + obase : nullptr;
    auto put = [&](int o, uint32_t w, int j) {
      const int idx = ES == 2 ? static_cast<int>(w >> 16) : static_cast<int>(ci[j]);
      if (IDX64) oi64[o] = idx;
      else oi32[o] = idx;
      if (RETV) ov[o] = static_cast<VT>(ES == 2 ? (w & 0xFFFFu) : w);
    };
    if (!p.ordered) {
      int o_gt = 0;
      for (int j0 = 0; j0 < n; j0 += 32 * kSelU) {
        uint32_t wv[kSelU];
#pragma unroll
        for (int u = 0; u < kSelU; ++u) {
          const int j = j0 + 32 * u + lane;
          wv[u] = j < n ? cw[j] : 0u;
        }
#pragma unroll
        for (int u = 0; u < kSelU; ++u) {
          const bool sel = j0 + 32 * u + lane < n && key_of<ES>(ES == 2 ? (wv[u] & 0xFFFFu) : wv[u]) > kth;
          const uint32_t sb = __ballot_sync(kFull, sel);
          if (sel) put(o_gt + __popc(sb & lt), wv[u], j0 + 32 * u + lane);
          o_gt += __popc(sb);
        }
      }
      int t_eq = 0;
      for (int j0 = 0; j0 < n && t_eq < static_cast<int>(need); j0 += 32) {
        const int j = j0 + lane;
        const uint32_t w = j < n ? cw[j] : 0u;
        const bool eq = j < n && key_of<ES>(ES == 2 ? (w & 0xFFFFu) : w) == kth;
        const uint32_t eb = __ballot_sync(kFull, eq);
        const int r = t_eq + __popc(eb & lt);
        if (eq && r < static_cast<int>(need)) put(o_gt + r, w, j);
        t_eq += __popc(eb);
      }
      return;
    }
    int taken_eq = 0, out = 0;
    for (int j0 = 0; j0 < n && out < p.k; j0 += 32 * kSelU) {
      uint32_t wv[kSelU], gtb[kSelU], eqb[kSelU];
#pragma unroll
      for (int u = 0; u < kSelU; ++u) {
        const int j = j0 + 32 * u + lane;
        wv[u] = j < n ? cw[j] : 0u;  // bf16: bits | index << 16; fp32: bits
      }
#pragma unroll
      for (int u = 0; u < kSelU; ++u) {
        const bool in = j0 + 32 * u + lane < n;
        const uint32_t key = key_of<ES>(ES == 2 ? (wv[u] & 0xFFFFu) : wv[u]);
        gtb[u] = __ballot_sync(kFull, in && key > kth);
        eqb[u] = __ballot_sync(kFull, in && key == kth);
      }
#pragma unroll
      for (int u = 0; u < kSelU; ++u) {
        const bool eq = (eqb[u] >> lane) & 1u;
        const bool sel = ((gtb[u] >> lane) & 1u) ||
                         (eq && static_cast<uint32_t>(taken_eq + __popc(eqb[u] & lt)) < need);
        taken_eq += __popc(eqb[u]);
        const uint32_t sb = __ballot_sync(kFull, sel);
        const int o = out + __popc(sb & lt);
        if (sel && o < p.k) put(o, wv[u], j0 + 32 * u + lane);
        out += __popc(sb);
      }
    }
  }

  // ---- R + C on the candidates ---------------------------------------------------
  // n candidates (k <= n <= cap), every non-NaN one with key >= tk, in index
  // order. Writes the row's top k and returns 1 with the k-th key in *kth, or
  // returns 0 (nothing written) if a candidate is NaN.
  __device__ int select_candidates(int64_t row, int n, uint32_t tk, uint32_t* kth_out) const {
    constexpr int S0 = KB - 16;  // the first level bins the top 16 key bits
    uint32_t need = static_cast<uint32_t>(p.k);
    const uint32_t lo16 = tk >> S0;
    wr_clear_hist(hist);
    uint32_t over = 0;
    bool nan = false;
    for (int j0 = 0; j0 < n; j0 += 32 * kSelU) {  // kSelU candidates per lane in flight
      uint32_t bits[kSelU];
#pragma unroll
      for (int u = 0; u < kSelU; ++u) {
        const int j = j0 + 32 * u + lane;
        bits[u] = j < n ? bits_at(j) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kSelU; ++u) {
        if (j0 + 32 * u + lane < n) {
          nan |= is_nan_bits<ES>(bits[u]);
          const uint32_t d = (key_of<ES>(bits[u]) >> S0) - lo16;
          if (d < 256u) atomicAdd(&hist[d], 1u);
          else ++over;
        }
      }
    }
    if (__any_sync(kFull, nan)) return 0;
    over = __reduce_add_sync(kFull, over);
    __syncwarp();
    uint32_t lo, hi;
    if (over < need) {  // the k-th key lies in the window
      uint32_t above, cnt;
      const uint32_t b = wr_find_bin(hist, need - over, &above, &cnt);
      __syncwarp();
      need -= over + above;
      lo = (lo16 + b) << S0;
      hi = lo + ((1u << S0) - 1u);
    } else {  // above it (t far below the k-th key): the range up to the largest key
      lo = (lo16 + 256u) << S0;
      hi = KB == 16 ? 0xFFFFu : 0xFFFFFFFFu;
    }
    while (lo < hi) {  // 8-bit levels over [lo, hi]
      const uint32_t span = hi - lo;
      const int s = span < 256u ? 0 : (32 - __clz(span)) - 8;
      wr_clear_hist(hist);
      for (int j = lane; j < n; j += 32) {
        const uint32_t key = key_of<ES>(bits_at(j));
        if (key >= lo && key <= hi) atomicAdd(&hist[(key - lo) >> s], 1u);
      }
      __syncwarp();
      uint32_t above, cnt;
      const uint32_t b = wr_find_bin(hist, need, &above, &cnt);
      __syncwarp();
      need -= above;
      lo += b << s;
      if (s == 0) break;
      const uint32_t top = lo + ((1u << s) - 1u);
      hi = top < hi ? top : hi;
    }
    const uint32_t kth = lo;
    // ordered output: ties (key == kth) are taken in index order, `need` of them
    if (p.idx64) {
      if (p.return_value) write_out<true, true>(row, n, kth, need);
      else write_out<true, false>(row, n, kth, need);
    } else {
      if (p.return_value) write_out<false, true>(row, n, kth, need);
      else write_out<false, false>(row, n, kth, need);
    }
    *kth_out = kth;
    return 1;
  }

  // ---- exact k-th largest vector maximum (top 16 key bits) --------------------------
  // Two passes over the row, one histogram update per vector. At least k
  // elements reach the result, so it is a threshold that always holds.
  __device__ uint32_t vecmax_threshold(const Geo& g) const {
    if (dense(g)) return elem_threshold(g, static_cast<uint32_t>(p.k), (g.nv + 31) / 32, 32);
    if (g.nv < p.k) return wr_key_floor<ES>();
    const int nsteps = (g.nv + 31) / 32;
    uint32_t need = static_cast<uint32_t>(p.k), b1 = 0;
    for (int level = 0; level < 2; ++level) {
      wr_clear_hist(hist);
      for (int i = 0; i < nsteps; ++i) {
        const int v = i * 32 + lane;
        if (v < g.nv) {
          const uint32_t kk = key16(vec_max<ES>(load(g, v)));
          if (level == 0) atomicAdd(&hist[kk >> 8], 1u);
          else if ((kk >> 8) == b1) atomicAdd(&hist[kk & 0xFFu], 1u);
        }
      }
      __syncwarp();
      uint32_t above, cnt;
      const uint32_t b = wr_find_bin(hist, need, &above, &cnt);
      __syncwarp();
      need -= above;
      if (level == 0) b1 = b;
      else b1 = (b1 << 8) | b;
    }
    uint32_t t = b1;
    if constexpr (ES == 4) t <<= 16;
    return t < wr_key_floor<ES>() ? wr_key_floor<ES>() : t;
  }

  // ---- exact fallback: radix levels over every element, then an ordered pass ------
  __device__ void exact_row(const Geo& g, int64_t row) const {
    const int nvec = g.nv;
    const int nsteps = (nvec + 31) / 32;
    uint32_t prefix = 0, need = static_cast<uint32_t>(p.k);
    bool nan = false;
    for (int done = 0; done < KB; done += 8) {
      wr_clear_hist(hist);
      const int sh = KB - done - 8;
      for (int i = 0; i < nsteps; ++i) {
        const int v = i * 32 + lane;
        if (v >= nvec) continue;
        const uint4 w = load(g, v);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const int idx = v * VEC + e - g.lead;
          if (idx >= 0 && idx < p.len) {
            const uint32_t bits = elem_bits<ES>(w, e);
            if (done == 0) nan |= is_nan_bits<ES>(bits);
            const uint32_t key = key_of<ES>(bits);
            if (done == 0 || (key >> (sh + 8)) == prefix) atomicAdd(&hist[(key >> sh) & 0xFFu], 1u);
          }
        }
      }
      __syncwarp();
      uint32_t above, cnt;
      const uint32_t b = wr_find_bin(hist, need, &above, &cnt);
      __syncwarp();
      need -= above;
      prefix = (prefix << 8) | b;
    }
    if (__any_sync(kFull, nan) && lane == 0) atomicOr(p.flag, DS_TOPK_FLAG_NAN);
    const uint32_t kth = prefix;
    int taken_eq = 0, out = 0;
    const int64_t obase = row * p.k;
    for (int i = 0; i < nsteps && out < p.k; ++i) {
      const int v = i * 32 + lane;
      uint4 w = make_uint4(0, 0, 0, 0);
      uint32_t mgt = 0, meq = 0;
      if (v < nvec) {
        w = load(g, v);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const int idx = v * VEC + e - g.lead;
          if (idx >= 0 && idx < p.len) {
            const uint32_t key = key_of<ES>(elem_bits<ES>(w, e));
            mgt |= static_cast<uint32_t>(key > kth) << e;
            meq |= static_cast<uint32_t>(key == kth) << e;
          }
        }
      }
      // ties before this lane's vector, in index order
      const uint32_t ce = __popc(meq);
      const uint32_t pe = warp_excl_scan(ce);
      const uint32_t te = __shfl_sync(kFull, pe + ce, 31);
      const int before = taken_eq + static_cast<int>(pe);
      int take = static_cast<int>(need) - before;
      take = take < 0 ? 0 : (take > static_cast<int>(ce) ? static_cast<int>(ce) : take);
      uint32_t msel = mgt;
      uint32_t mq = meq;
      for (int t = 0; t < take; ++t) {
        msel |= mq & (0u - mq);  // lowest remaining tie
        mq &= mq - 1;
      }
      taken_eq += static_cast<int>(te);
      const uint32_t cs = __popc(msel);
      const uint32_t ps = warp_excl_scan(cs);
      const int ts = static_cast<int>(__shfl_sync(kFull, ps + cs, 31));
      int64_t o = obase + out + ps;
      while (msel && o < obase + p.k) {
        const int e = __ffs(msel) - 1;
        msel &= msel - 1;
        put_index(p.out_indices, o, v * VEC + e - g.lead, p.idx64);
        if (p.return_value) {
          const uint32_t bits = elem_bits<ES>(w, e);
          if constexpr (ES == 2) static_cast<uint16_t*>(p.out_values)[o] = static_cast<uint16_t>(bits);
          else static_cast<uint32_t*>(p.out_values)[o] = bits;
        }
        ++o;
      }
      out += ts;
    }
  }
};

// Margin (in top-16 key units) below the previous row's k-th key for the next
// row's threshold guess. Measured on the decode-shaped call: 8 is fastest (4, 5
// and 6 cost more failed guesses and their retries, 10 to 16 more candidates).
constexpr uint32_t kWrGuessMargin = 8;

template <int ES>
__global__ void __launch_bounds__(kWrThreads, 3) topk_warp_rows_kernel(const WrParams p) {
  // let the next kernel in the stream start its prologue; wait for the previous one
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const WarpRow<ES> wr(p, smem + warp * wr_warp_bytes(ES, p.cap, p.depth));
  constexpr int KB = Traits<ES>::kKeyBits;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWrWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWrWarps + warp;
  if (wr.lane == 0) {
    for (int i = 0; i < p.depth; ++i) mbar_init(wr.mbar + i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();
  // the warp's rows stream through its ring back to back: the next row's first
  // chunks are in flight while the current row is being selected
  typename WarpRow<ES>::Stream st;
  wr.stream_begin(st, first);
  for (int i = 0; i < p.depth; ++i) wr.produce_one(st, nwarps);
  bool have_guess = false;
  uint32_t guess = 0;
  for (int64_t row = first; row < p.batch; row += nwarps) {
    const typename WarpRow<ES>::Geo g = wr.geo(row);
    uint32_t q = 0;
    uint32_t tk = have_guess ? guess : wr.sample_threshold(g, q = wr.default_rank(g));
    int n = 0;
    if (!wr.stream_pass(st, nwarps, g, tk, &n)) {
      if (wr.lane == 0) atomicOr(p.flag, DS_TOPK_FLAG_TIMEOUT);
      wr.drain(st);
      return;
    }
    // 1: selected; 0: a NaN among the candidates; -1: the guess did not hold
    uint32_t kth = 0;
    int status = (n >= p.k && n <= p.cap) ? wr.select_candidates(row, n, tk, &kth) : -1;
    // retries, each a direct pass over the row (from L2): the default sample
    // rank after a carried guess, then a rank adapted to the count just seen,
    // then the exact k-th largest vector maximum
    for (int attempt = have_guess ? 0 : 1; status < 0 && attempt < 3; ++attempt) {
      if (attempt == 0) q = wr.default_rank(g);
      if (attempt == 1) q = wr.adapted_rank(q, n);
      tk = attempt == 2 ? wr.vecmax_threshold(g) : wr.sample_threshold(g, q);
      n = wr.direct_pass(g, tk);
      if (n >= p.k && n <= p.cap) status = wr.select_candidates(row, n, tk, &kth);
    }
    if (status == 1) {
      const uint32_t m = (KB == 16 ? kWrGuessMargin : (kWrGuessMargin << 16));
      guess = kth > wr_key_floor<ES>() + m ? kth - m : wr_key_floor<ES>();
      have_guess = true;
    } else {
      wr.exact_row(g, row);  // also raises the NaN flag
    }
    __syncwarp();
  }
}

}  // namespace ds_topk_dev
