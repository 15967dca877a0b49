// chain_stochastic.cu -- the stochastic chain verifier.
//
// Computes the test of "Speculative Decoding: Draft, Verify, and Correct"
// ('Name the two distributions at one prefix', 'Verify several proposed tokens
// in one target pass'): p = softmax(target/T), q = softmax(draft/T); position
// j accepts y_j iff p(y_j)/q(y_j) >= 1 or u < p(y_j)/q(y_j); the walk stops at
// the first rejection and draws the correction from the residual [p - q]+ by
// inverse CDF; if every draft passes, the bonus token is drawn from p_K.
//
// The plain verify runs two kernels per call after a one-thread step that
// advances the workspace's generation (the stamp every record of the call
// carries).  Each of the three is a programmatic dependent of the kernel
// before it; the generation step lets the stream start only once every
// earlier kernel has completed, and no kernel touches the workspace before
// the generation step itself has.
//
//  softmax_partials_kernel -- the HBM stream.  A persistent grid (several CTAs
//    per SM, no clusters) walks (logit row, vocabulary slice) items through a
//    bulk-copy (TMA) ring in shared memory.  Each item yields the slice's max
//    logit m and sum of exp2((x - m) log2(e) / T) (an online softmax: each
//    thread exponentiates against its own max, warps and the CTA fold the
//    pairs) and, if the slice holds the draft token, its logit.  Every logit
//    is read from HBM exactly once here, with one exp per logit.  Positions
//    j >= 2 are streamed first and positions 0 and 1 last, loaded without the
//    evict-first hint when they fit well inside L2, so the rows where walks
//    most often stop are still there for the second kernel.
//
//  chain_resolve_kernel -- one thread-block cluster per batch row, launched as
//    a programmatic dependent of the first kernel.  Every CTA of the cluster
//    polls the row's stamped partials, folds them into the global max and sum
//    of each position, forms the acceptance ratios in log2 space and finds the
//    first rejection (the same arithmetic in every CTA gives the same bits).
//    The cluster then re-reads only the stopping position (the residual needs
//    the global normalisers, so it cannot be formed during the stream): each
//    CTA sums the residual mass of its vocabulary slice, one cluster barrier
//    exchanges the masses, and the CTA, warp, round, lane and element whose
//    cumulative interval holds u * mass are chosen in vocabulary order.
//
// The truncated verify lets the stream also keep, per truncated logit row,
// the maximum of every consumer thread's chunk of each tile, and selects each
// row's top-k / top-p thresholds from the chunks those maxima point to (one
// CTA per logit row) ahead of the same resolve kernel.  DRIFT residuals run
// the stream over positions 0 .. K-1 (chunk maxima for the target rows),
// drift_pick_kernel (one CTA per drafted position: the top m of its target
// row from those chunks) and drift_finish_kernel (one CTA per row: log q at
// the support, the residuals and the row status).
#include <cuda_bf16.h>

#include <atomic>
#include <cstddef>

#include "common.cuh"
#include "internal.h"
#include "specverify.h"

namespace sv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kInf = __builtin_huge_valf();
constexpr int kMaxStages = 4;

template <bool BF16>
struct Fmt {
  static constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr uint32_t NEG_INF_WORD = BF16 ? 0xFF80FF80u : 0xFF800000u;
  static __device__ __forceinline__ float elem(const uint32_t *w, int e) {
    if constexpr (BF16) return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
    else return __uint_as_float(w[e]);
  }
  // elements 2i and 2i+1 of a 16-byte vector
  static __device__ __forceinline__ float2 pair(const uint32_t *w, int i) {
    if constexpr (BF16) return make_float2(bf16_lo(w[i]), bf16_hi(w[i]));
    else return make_float2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
  }
  static __device__ __forceinline__ void mask_tail(uint32_t *w, int valid) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      if (e >= valid) {
        if constexpr (BF16) {
          w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0x0000ffffu) | 0xFF800000u)
                              : ((w[e >> 1] & 0xffff0000u) | 0x0000FF80u);
        } else {
          w[e] = 0xFF800000u;
        }
      }
    }
  }
  // Vector v of a slice of `len` elements starting at gsrc: from a shared-
  // memory copy (sbuf != nullptr), else from global memory (16-byte loads when
  // `aligned`, element loads otherwise).  Elements >= len read as -inf.
  static __device__ __forceinline__ void load_vec(uint32_t *w, const unsigned char *sbuf,
                                                  const char *gsrc, bool aligned, int v, int len) {
    const int valid = len - v * EPV;
    if (valid <= 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = NEG_INF_WORD;
      return;
    }
    if (sbuf) {
      const uint4 r = ld_shared_u4(sbuf + (size_t)v * 16);
      w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    } else if (aligned) {
      const uint4 r = __ldg(reinterpret_cast<const uint4 *>(gsrc) + v);
      w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
          const int e0 = v * 8 + 2 * i;
          const unsigned short *g = reinterpret_cast<const unsigned short *>(gsrc);
          const uint32_t lo = e0 < len ? __ldg(g + e0) : 0xFF80u;
          const uint32_t hi = e0 + 1 < len ? __ldg(g + e0 + 1) : 0xFF80u;
          w[i] = lo | (hi << 16);
        } else {
          const int e = v * 4 + i;
          w[i] = e < len ? __ldg(reinterpret_cast<const unsigned int *>(gsrc) + e) : 0xFF800000u;
        }
      }
    }
    if (valid < EPV) mask_tail(w, valid);
  }
};

// Fold (max, sum relative to that max) pairs across the lanes of a warp in a
// fixed butterfly order; every lane gets the result.  -inf maxima carry no mass.
__device__ __forceinline__ void fold_max_sum(float m, float s, float s2, float *Mout, float *Sout) {
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmax_nan(M, __shfl_xor_sync(FULL_MASK, M, o));
  float v = (m == -kInf || s == 0.f) ? 0.f : s * ex2(__fmul_rn(m - M, s2));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  *Mout = M;
  *Sout = v;
}

// The first of n entries (lane c holds entry c's mass, in order) whose
// cumulative interval holds t; past the total it clamps to the last positive
// entry.  Returns the entry and the remainder inside it (+inf when clamped),
// or -1 without mass.
__device__ __forceinline__ int pick_entry(float mass_lane, int n, float t, float *t_in) {
  float acc = 0.f, tl = kInf;
  int cs = -1, clast = -1;
  for (int c = 0; c < n; ++c) {
    const float m = __shfl_sync(FULL_MASK, mass_lane, c);
    const float prev = acc;
    acc += m;
    if (m > 0.f) {
      clast = c;
      if (cs < 0 && acc > t) {
        cs = c;
        tl = t - prev;
      }
    }
  }
  if (cs < 0) {
    cs = clast;
    tl = kInf;
  }
  *t_in = tl;
  return cs;
}

__device__ __forceinline__ float sum_lanes(float v, int n) {
  float s = 0.f;
  for (int c = 0; c < n; ++c) s += __shfl_sync(FULL_MASK, v, c);
  return s;
}

// ============================================================ kernel 1

// Per-tile facts every consumer needs, computed by the producer warp and
// kept next to the tile's stage.  A tile is the same vocabulary range of a
// position's target row and (for j < K) its draft row, streamed together so
// that both laws see the same arithmetic.
struct alignas(16) TileInfo {
  long long tsrc;  // byte offset of the target tile
  long long dsrc;  // byte offset of the draft tile (pair tiles only)
  int trow;        // partial row of the target row
  int drow;        // partial row of the draft row, -1 for the bonus position
  int run0;        // tile index (within the row) where this run of tiles starts
  int t;           // tile index within the row
  int len;         // elements in the tile
  int yl;          // tile index of the draft token, -1 if not here
  float s2;        // log2(e) / T
  int keep;        // 1: load without the evict-first hint
  int first;       // 1: first tile of a run
  int last;        // 1: last tile of a run
  int sketch;      // truncated verify: 1 = store the tile's chunk maxima
};

struct alignas(16) SoftCtrl {
  uint64_t full[kMaxStages];   // stage s holds its tile (producer -> consumers)
  uint64_t empty[kMaxStages];  // every consumer warp has copied stage s (consumers -> producer)
  uint64_t never;              // a barrier nothing completes (forced-timeout test)
  int broken;                  // a wait gave up: stop the pipeline
  int pad0;
  TileInfo info[kMaxStages];   // facts of the tile in stage s
  float4 wpart[2 * kMaxStages][kSoftThreads / 32];  // per-warp (max p, sum p, max q, sum q), by run
  uint32_t tflags[2 * kMaxStages];                  // timeout seen, by run
  int arrived[2 * kMaxStages];                      // warps done, by run
};
static_assert(sizeof(SoftCtrl) <= 2048, "control block must fit its reservation");

// Positions in stream order: the bonus positions (j = K), then j = K-1 down
// to 2, each over b = 0..B-1; then positions 1 and 0 row by row.
__device__ __forceinline__ void stream_pos(int i, int B, int K, int *b, int *j) {
  const int pa = K >= 2 ? B * (K - 1) : 0;
  if (i < pa) {  // positions K .. 2, each over every row
    *j = K - i / B;
    *b = i - (K - *j) * B;
  } else {       // the rest row by row, so rows complete one after another
    const int npb = K >= 2 ? 2 : K + 1;
    const int i2 = i - pa;
    *b = i2 / npb;
    *j = npb - 1 - (i2 - *b * npb);
  }
}

// Order-preserving integer key of a logit's raw bits (larger logit, larger
// key; -inf smallest).
template <bool BF16>
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  if constexpr (BF16) return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
  else return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// Raw bits of element e of a 16-byte vector.
template <bool BF16>
__device__ __forceinline__ uint32_t elem_bits(const uint32_t *w, int e) {
  if constexpr (BF16) return (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
  else return w[e];
}

// The logit value whose order key is k (inverse of order_key).
template <bool BF16>
__device__ __forceinline__ float key_value(uint32_t k) {
  if constexpr (BF16) {
    const uint32_t bits = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(bits << 16);
  } else {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  }
}

// Bit e is set for each element e of a 16-byte vector that is not below the
// threshold value tf (tw: tf's bf16 bits in both halves, for bf16).  Every
// element whose order key reaches the threshold's has a value >= tf, so a
// clear bit is exact; a NaN element or threshold sets the bit.
template <bool BF16>
__device__ __forceinline__ uint32_t may_reach_bits(const uint32_t *w, uint32_t tw, float tf) {
  uint32_t bits = 0;
  if constexpr (BF16) {
    const __nv_bfloat162 t2 = *reinterpret_cast<const __nv_bfloat162 *>(&tw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t ge = ~__hlt2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]), t2);
      bits |= ((ge & 1u) | ((ge >> 15) & 2u)) << (2 * i);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) bits |= (__uint_as_float(w[i]) < tf ? 0u : 1u) << i;
  }
  return bits;
}

// Raw bits of element e (a run-time index) of a 16-byte vector held in
// registers: the word is chosen by selects, not by indexing.
template <bool BF16>
__device__ __forceinline__ uint32_t elem_bits_at(const uint32_t *w, int e) {
  const int i = BF16 ? (e >> 1) : e;
  const uint32_t x = i < 2 ? (i == 0 ? w[0] : w[1]) : (i == 2 ? w[2] : w[3]);
  if constexpr (BF16) return (e & 1) ? (x >> 16) : (x & 0xFFFFu);
  else return x;
}

// The threshold value tf's bf16 bits in both halves of a word (any value for fp32).
template <bool BF16>
__device__ __forceinline__ uint32_t pack_threshold(float tf) {
  if constexpr (BF16) {
    const uint32_t hb = __float_as_uint(tf) >> 16;
    return hb | (hb << 16);
  } else {
    return 0u;
  }
}

// The row's top-k / top-p parameters; false when neither truncates.
__device__ __forceinline__ bool trunc_active(const ChainStochParams &P, int b, int V, int *k,
                                             float *tp) {
  *k = P.top_k ? P.top_k[b] : 0;
  *tp = P.top_p ? P.top_p[b] : 1.0f;
  const bool use_k = *k >= 1 && *k < V;
  const bool use_p = *tp > 0.f && *tp < 1.f;
  if (!use_k) *k = 0;
  if (!use_p) *tp = 1.0f;
  return use_k || use_p;
}

// Stamped partial records (see SoftPart).
__device__ __forceinline__ void store_part(SoftPart *d, float m, float s, uint32_t flags, uint32_t tag) {
  st_relaxed_u64(&d->a, static_cast<unsigned long long>(__float_as_uint(m)) |
                            (static_cast<unsigned long long>(tag) << 32));
  st_relaxed_u64(&d->b, static_cast<unsigned long long>(__float_as_uint(s)) |
                            (static_cast<unsigned long long>((flags & 0xffu) | (tag << 8)) << 32));
}
// A record's two words, decoded; false while either holds an older record.
__device__ __forceinline__ bool decode_part(unsigned long long a, unsigned long long b, uint32_t tag,
                                            float *m, float *s, uint32_t *flags) {
  *m = __uint_as_float(static_cast<uint32_t>(a));
  *s = __uint_as_float(static_cast<uint32_t>(b));
  const uint32_t hb = static_cast<uint32_t>(b >> 32);
  *flags = hb & 0xffu;
  return static_cast<uint32_t>(a >> 32) == tag && (hb >> 8) == (tag & 0xffffffu);
}
// false while either word still holds an older record
__device__ __forceinline__ bool load_part(const SoftPart *d, uint32_t tag, float *m, float *s,
                                          uint32_t *flags) {
  const unsigned long long a = ld_relaxed_u64(&d->a), b = ld_relaxed_u64(&d->b);
  *m = __uint_as_float(static_cast<uint32_t>(a));
  *s = __uint_as_float(static_cast<uint32_t>(b));
  const uint32_t hb = static_cast<uint32_t>(b >> 32);
  *flags = hb & 0xffu;
  return static_cast<uint32_t>(a >> 32) == tag && (hb >> 8) == (tag & 0xffffffu);
}

// Element offset of partial row `row` (targets b*(K+1)+j, then drafts
// B*(K+1) + b*K + j) in its logits tensor.
__device__ __forceinline__ long long row_offset(const ChainStochParams &P, int row) {
  const int npos = P.K + 1;
  return row < P.B * npos ? (long long)row * P.V : (long long)(row - P.B * npos) * P.V;
}

// A phase is a range of positions [p0, p1) of the stream; its tiles cost 1
// (bonus position: target only) or 2 (target and draft).  Returns the first
// tile (phase-relative) of CTA g's even share of the phase's cost.
__device__ __forceinline__ int phase_split(int p0, int p1, int B, int K, int nt, int g, int G) {
  const int nb = max(0, min(p1, B) - p0) * nt;     // bonus tiles (they come first)
  const int np = (p1 - p0) * nt - nb;              // pair tiles
  const long long cost = (long long)nb + 2LL * np;
  const long long c = cost * g / G;
  return c <= nb ? (int)c : nb + (int)((c - nb + 1) / 2);
}

template <bool BF16, bool CAND>
__device__ __forceinline__ TileInfo make_tile(const ChainStochParams &P, int gt, int lo, int hi) {
  TileInfo it;
  const int B = P.B, K = P.K, nt = P.nslices;
  const int i = gt / nt;
  it.t = gt - i * nt;
  int b, j;
  stream_pos(i, B, P.drift_m > 0 ? K - 1 : K, &b, &j);  // DRIFT: no bonus position
  const int s0 = it.t * P.slice;
  it.len = min(P.V - s0, P.slice);
  it.trow = b * (K + 1) + j;
  it.tsrc = ((long long)it.trow * P.V + s0) * Fmt<BF16>::ESZ;
  if (j < K) {
    it.drow = B * (K + 1) + b * K + j;
    it.dsrc = ((long long)(b * K + j) * P.V + s0) * Fmt<BF16>::ESZ;
  } else {
    it.drow = -1;
    it.dsrc = 0;
  }
  it.keep = j < P.keep_pos;
  // a run is the part of a row inside [lo, hi): it starts at the later of lo
  // and the row's first tile
  it.first = (gt == lo) || it.t == 0;
  it.last = (gt == hi - 1) || it.t == nt - 1;
  it.run0 = max(lo - (gt - it.t), 0);
  float T = P.temperature && SV_INB(b, B) ? __ldg(P.temperature + b) : 1.0f;
  if (!(T > 0.f && T < kInf)) T = 1.0f;  // the resolve kernel flags the row
  it.s2 = __fdiv_rn(kLog2e, T);
  it.yl = -1;
  if (j < K && P.tokens && SV_INB((long long)b * K + j, (long long)B * K)) {
    const int y = __ldg(P.tokens + (size_t)b * K + j);
    if (y >= s0 && y < s0 + it.len) it.yl = y - s0;
  }
  it.sketch = 0;
  if constexpr (CAND) {
    int tk;
    float tp;
    it.sketch = P.drift_m > 0 || (SV_INB(b, B) && trunc_active(P, b, P.V, &tk, &tp));
  }
  return it;
}

// The n-th tile of the CTA, rebuilt by a consumer after a wait gave up.
template <bool BF16, bool CAND>
__device__ __noinline__ TileInfo rebuild_tile(const ChainStochParams &P, int n, int na, int lo_a,
                                              int hi_a, int lo_b, int hi_b) {
  return n < na ? make_tile<BF16, CAND>(P, lo_a + n, lo_a, hi_a)
                : make_tile<BF16, CAND>(P, lo_b + (n - na), lo_b, hi_b);
}

template <bool BF16, int NV>
__device__ __forceinline__ void load_tile(uint32_t (&w)[NV * 4], bool tma, uint32_t sbase,
                                          const char *gsrc, int tid, int nvec, int len) {
  using F = Fmt<BF16>;
  if (tma) {  // whole 16-byte vectors: tiles are multiples of 8 bf16 / 4 fp32 here
    const uint32_t a = sbase + tid * 16;
    if (nvec == NV * kSoftThreads) {
#pragma unroll
      for (int k = 0; k < NV; ++k)
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[4 * k]), "=r"(w[4 * k + 1]), "=r"(w[4 * k + 2]), "=r"(w[4 * k + 3])
                     : "r"(a + k * kSoftThreads * 16));
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (tid + k * kSoftThreads < nvec) {
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[4 * k]), "=r"(w[4 * k + 1]), "=r"(w[4 * k + 2]), "=r"(w[4 * k + 3])
                       : "r"(a + k * kSoftThreads * 16));
        } else {
          w[4 * k] = w[4 * k + 1] = w[4 * k + 2] = w[4 * k + 3] = F::NEG_INF_WORD;
        }
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < NV; ++k) F::load_vec(w + 4 * k, nullptr, gsrc, false, tid + k * kSoftThreads, len);
  }
}

template <bool BF16, int NV>
__device__ __forceinline__ float tile_max(const uint32_t (&w)[NV * 4]) {
  using F = Fmt<BF16>;
  if constexpr (BF16) {
    uint32_t pm0 = F::NEG_INF_WORD, pm1 = F::NEG_INF_WORD;
#pragma unroll
    for (int i = 0; i < NV * 4; i += 2) {
      pm0 = bf16x2_max_nan(pm0, w[i]);
      pm1 = bf16x2_max_nan(pm1, w[i + 1]);
    }
    pm0 = bf16x2_max_nan(pm0, pm1);
    return fmax_nan(bf16_lo(pm0), bf16_hi(pm0));
  } else {
    float m0 = -kInf, m1 = -kInf;
#pragma unroll
    for (int i = 0; i < NV * 4; i += 2) {
      m0 = fmax_nan(m0, __uint_as_float(w[i]));
      m1 = fmax_nan(m1, __uint_as_float(w[i + 1]));
    }
    return fmax_nan(m0, m1);
  }
}

// Fold one tile into a running (max, sum of exp2((x - max) s2)); element
// pairs through packed fp32 (one fma and one add per pair).  Returns the
// largest of the thread's elements of the tile.
template <bool BF16, int NV>
__device__ __forceinline__ float tile_accumulate(const uint32_t (&w)[NV * 4], float s2, int tid,
                                                 int nvec, float &m_run, float &s_run) {
  using F = Fmt<BF16>;
  const float m = tile_max<BF16, NV>(w);
  const float m_new = fmax_nan(m_run, m);
  if (m_run != -kInf && m_new != m_run) s_run *= ex2(__fmul_rn(m_run - m_new, s2));
  m_run = m_new;
  const float off = (m_run == -kInf) ? 0.f : -__fmul_rn(m_run, s2);
  const float2 s2v = make_float2(s2, s2), offv = make_float2(off, off);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);  // independent chains
  const bool full = nvec == NV * kSoftThreads;  // no bounds
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (full || tid + k * kSoftThreads < nvec) {
#pragma unroll
      for (int i = 0; i < F::EPV / 2; ++i) {
        const float2 a = ffma2(F::pair(w + 4 * k, i), s2v, offv);
        const float2 e = make_float2(ex2(a.x), ex2(a.y));
        if (i & 1) acc1 = fadd2(acc1, e);
        else acc0 = fadd2(acc0, e);
      }
    }
  }
  s_run += (acc0.x + acc0.y) + (acc1.x + acc1.y);
  return m;
}

// Warp-specialised stream.  Each CTA owns one contiguous share (even in cost)
// of the tiles of phase A (positions >= 2) and one of phase B (positions 0
// and 1, streamed last so they stay in L2 for the resolve kernel).  Warp NW
// (the producer) walks them in order, writes each tile's facts next to its
// stage and issues the bulk copies; warps 0..NW-1 (the consumers) take the
// tile into registers, release the stage, and fold it into a running (max,
// sum) per thread and per law: a run of tiles of one position costs one
// rescale per tile and a single CTA-wide fold at its end.  Producer and
// consumers meet only on the full/empty barriers of each stage.
//
// With CAND (the truncated verify) each consumer thread also stores, for a
// truncated row, the largest of its elements of the tile (its "chunk": 4
// vectors, 32 bf16 or 16 fp32 logits), which the fold computes anyway: one
// 2-byte store per chunk, 1/16 of the bf16 logit bytes.
template <bool BF16, int NV, int S, bool CAND>
__global__ void __launch_bounds__(kSoftThreads + 32, kSoftMinBlocks) softmax_partials_kernel(const __grid_constant__ ChainStochParams P) {
  using F = Fmt<BF16>;
  constexpr int NT = kSoftThreads, NW = NT / 32;
  constexpr int EPV = F::EPV, ESZ = F::ESZ;
  extern __shared__ __align__(128) unsigned char smem[];
  SoftCtrl &ctl = *reinterpret_cast<SoftCtrl *>(smem + (size_t)S * P.buf_bytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = P.nslices, B = P.B, K = P.K;
  // DRIFT streams positions 0 .. K-1 only (every tile a pair): the stream
  // order of a chain with K-1 drafts, over the real rows
  const int Ks = P.drift_m > 0 ? K - 1 : K;
  const int npos = B * (Ks + 1);
  const int pa = Ks >= 2 ? B * (Ks - 1) : 0;  // positions with j >= 2 come first
  const int G = (int)gridDim.x, g = (int)blockIdx.x;
  const int lo_a = phase_split(0, pa, B, Ks, nt, g, G);
  const int hi_a = phase_split(0, pa, B, Ks, nt, g + 1, G);
  const int lo_b = pa * nt + phase_split(pa, npos, B, Ks, nt, g, G);
  const int hi_b = pa * nt + phase_split(pa, npos, B, Ks, nt, g + 1, G);
  // Only phase A is split statically; the tiles of phase B are claimed in
  // chunks (through the counter the generation step clears) as CTAs run out
  // of work, so CTAs that stream faster take more of the tail.
  const bool dyn = P.stream_dyn != 0;
  const int dyn_from = pa * nt;
  const int na = hi_a - lo_a;
  const int my_tiles = dyn ? na : na + (hi_b - lo_b);  // statically assigned tiles
  auto tile_of = [&](int n, int *lo, int *hi) {  // n-th static tile of this CTA
    if (n < na) {
      *lo = lo_a;
      *hi = hi_a;
      return lo_a + n;
    }
    *lo = lo_b;
    *hi = hi_b;
    return lo_b + (n - na);
  };
  const bool tma = P.use_tma != 0;
  const int half = P.buf_bytes / 2;  // target half, then draft half of a stage

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], NW);
    }
    mbar_init(&ctl.never, 1);
    ctl.broken = 0;
    for (int i = 0; i < 2 * kMaxStages; ++i) {
      ctl.arrived[i] = 0;
      ctl.tflags[i] = 0;
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NW) {  // ---------------------------------------------- producer
    if (lane != 0) return;
    const uint64_t pol_first = l2_policy_evict_first();
    const uint64_t pol_normal = l2_policy_evict_normal();
    int issued = 0;  // stages posted, the end marker included
    // wait until stage issued % S is free; false once the pipeline is broken
    auto next_stage = [&]() {
      const int s = issued % S;
      if (issued >= S &&
          !mbar_wait_bounded(&ctl.empty[s], static_cast<uint32_t>(issued / S - 1) & 1u, P.wait_limit_ns))
        ctl.broken = 1;
      return !*reinterpret_cast<volatile int *>(&ctl.broken);
    };
    auto post = [&](int gt, int lo, int hi) {
      if (!next_stage()) return false;
      const int s = issued % S;
      const TileInfo it = make_tile<BF16, CAND>(P, gt, lo, hi);
      ctl.info[s] = it;
      if (tma) {
        const uint32_t bytes = static_cast<uint32_t>(it.len) * ESZ;
        const uint64_t pol = it.keep ? pol_normal : pol_first;
        mbar_arrive_expect_tx(&ctl.full[s], it.drow >= 0 ? 2 * bytes : bytes);  // release: info[s] too
        // (bounds build: a copy out of range is skipped; its consumers time out)
        if (SV_INR(it.tsrc, bytes, (long long)B * (K + 1) * P.V * ESZ) &&
            SV_INR((long long)s * P.buf_bytes, bytes, (long long)S * P.buf_bytes))
          bulk_g2s(smem + (size_t)s * P.buf_bytes, static_cast<const char *>(P.target) + it.tsrc,
                   bytes, &ctl.full[s], pol);
        if (it.drow >= 0 && SV_INR(it.dsrc, bytes, (long long)B * K * P.V * ESZ) &&
            SV_INR((long long)s * P.buf_bytes + half, bytes, (long long)S * P.buf_bytes))
          bulk_g2s(smem + (size_t)s * P.buf_bytes + half,
                   static_cast<const char *>(P.draft) + it.dsrc, bytes, &ctl.full[s], pol);
      } else {
        mbar_arrive(&ctl.full[s]);
      }
      ++issued;
      return true;
    };
    bool ok = true;
    for (int n = 0; n < my_tiles && ok; ++n) {
      int lo, hi;
      const int gt = tile_of(n, &lo, &hi);
      ok = post(gt, lo, hi);
    }
    if (dyn && ok) {
      const int total = npos * nt;
      const int nchunks = (total - dyn_from + P.dyn_chunk - 1) / P.dyn_chunk;
      // A chunk is claimed only when the previous one is down to its last
      // tile, so no CTA holds more of the tail than its ring can take; the
      // claim's round trip overlaps the wait for that tile's stage.  The
      // counter is this call's once the generation step has completed.
      grid_dependency_wait();
      uint32_t claim = atomicAdd(P.claim, 1u);
      while (ok && claim < static_cast<uint32_t>(nchunks)) {
        const int lo = dyn_from + static_cast<int>(claim) * P.dyn_chunk;
        const int hi = min(lo + P.dyn_chunk, total);
        for (int gt = lo; gt < hi && ok; ++gt) {
          if (gt == hi - 1) claim = atomicAdd(P.claim, 1u);
          ok = post(gt, lo, hi);
        }
      }
    }
    if (ok && next_stage()) {  // end marker: a stage with no data
      const int s = issued % S;
      ctl.info[s].len = -1;
      mbar_arrive(&ctl.full[s]);
      ++issued;
    }
    // copies still landing after a give-up: wait (bounded) for the last phase
    // of every stage before leaving
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + ((issued - 1 - s) / S) * S;
      mbar_wait_bounded(&ctl.full[s], static_cast<uint32_t>(last / S) & 1u, P.wait_limit_ns);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  float mp = -kInf, sp = 0.f, mq = -kInf, sq = 0.f;  // running (max, sum) of p and q
  uint32_t run_to = 0;  // a timeout met in the current run (warp-uniform)
  int runs = 0;         // runs finished so far
  int s = 0;
  uint32_t parity = 0;
  const uint32_t smem0 = smem_u32(smem);
  // This grid is a programmatic dependent of the generation step and may
  // start before that step has written the tag.  Loading and folding tiles
  // needs nothing from it; a thread waits for it to complete just before its
  // first store to the workspace, and only then lets the resolve kernel,
  // which reads the tag as it starts, be scheduled.
  uint32_t tag = 0;
  bool joined = false;
  auto join_generation = [&]() {
    if (!joined) {
      grid_dependency_wait();
      tag = *reinterpret_cast<volatile const uint32_t *>(P.gen);
      allow_dependents();
      joined = true;
    }
  };
  // CAND: the chunk maximum of this thread's vectors of one row's tile, as
  // the top 16 bits of its order key, for the selection kernel
  auto store_chunk_max = [&](float m, int row, int t) {
    const long long at = ((long long)row * nt + t) * NT + tid;
    if (SV_INB(at, (long long)(2 * K + 1) * B * nt * NT))
      P.cmax[at] = static_cast<unsigned short>(order_key<false>(__float_as_uint(m)) >> 16);
  };
  // Stages arrive in the producer's order until its end marker (len < 0).
  for (int n = 0;; ++n, s = (s + 1 == S) ? 0 : s + 1, parity ^= (s == 0)) {
    bool timed_out = false;
    if (!*reinterpret_cast<volatile int *>(&ctl.broken)) {
      timed_out = P.force_timeout ? !mbar_wait_bounded(&ctl.never, 0u, P.wait_limit_ns)
                                  : !mbar_wait_bounded(&ctl.full[s], parity, P.wait_limit_ns);
    } else {
      timed_out = true;  // the pipeline stopped: this tile's data never came
    }
    timed_out = __any_sync(FULL_MASK, timed_out);
    // The facts next to the stage are only valid once its barrier completed.
    // After a give-up a statically assigned tile is rebuilt (the stage data is
    // then garbage but every index stays in bounds, and the row is flagged); a
    // claimed tile cannot be named, so the warp stops and that tile's records
    // keep an old stamp, which the resolve kernel reports as a timeout.
    TileInfo it;
    if (timed_out) {
      if (n >= my_tiles) break;
      it = rebuild_tile<BF16, CAND>(P, n, na, lo_a, hi_a, lo_b, hi_b);
    } else {
      it = ctl.info[s];
      if (it.len < 0) break;  // end marker
    }
    const bool pair = it.drow >= 0;
    const unsigned char *sb = smem + (size_t)s * P.buf_bytes;
    const int nvec = (it.len + EPV - 1) / EPV;
#ifdef SV_BOUNDS
    // the tile's vectors in the stage, its elements in the logit tensors, its
    // rows' records; the warp stops at a bad tile (its records stay
    // unwritten and their rows time out)
    {
      const bool ok = SV_INB(s, kMaxStages) && SV_INR(it.tsrc / ESZ, it.len, (long long)B * (K + 1) * P.V) &&
                      (!pair || SV_INR(it.dsrc / ESZ, it.len, (long long)B * K * P.V)) &&
                      (!tma || SV_INR((long long)s * P.buf_bytes, (long long)nvec * 16 + (pair ? half : 0),
                                      (long long)S * P.buf_bytes)) &&
                      SV_INR((long long)it.trow * nt + it.run0, it.t - it.run0 + 1,
                             (long long)(2 * K + 1) * B * nt) &&
                      (!pair || SV_INR((long long)it.drow * nt + it.run0, it.t - it.run0 + 1,
                                       (long long)(2 * K + 1) * B * nt));
      if (!__all_sync(FULL_MASK, ok)) break;
    }
#endif

    const uint32_t sbase = smem0 + s * P.buf_bytes;
    uint32_t wp[NV * 4];
    load_tile<BF16, NV>(wp, tma, sbase, static_cast<const char *>(P.target) + it.tsrc, tid, nvec, it.len);
    if (it.yl >= 0 && tid == 0 && SV_INB(it.yl, it.len) && SV_INB(it.trow, (2 * K + 1) * B) &&
        SV_INB(it.drow, (2 * K + 1) * B)) {  // the draft token's logits, if this tile holds them
      float a, c;
      if (tma) {
        const unsigned char *pv = sb + (size_t)it.yl * ESZ;
        if constexpr (BF16) {
          a = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short *>(pv)) << 16);
          c = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short *>(pv + half)) << 16);
        } else {
          a = *reinterpret_cast<const float *>(pv);
          c = *reinterpret_cast<const float *>(pv + half);
        }
      } else {
        const char *tg = static_cast<const char *>(P.target) + it.tsrc;
        const char *dg = static_cast<const char *>(P.draft) + it.dsrc;
        if constexpr (BF16) {
          a = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(tg) + it.yl)) << 16);
          c = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(dg) + it.yl)) << 16);
        } else {
          a = __ldg(reinterpret_cast<const float *>(tg) + it.yl);
          c = __ldg(reinterpret_cast<const float *>(dg) + it.yl);
        }
      }
      join_generation();
      st_relaxed_u64(P.ylog + it.trow, __float_as_uint(a) | (static_cast<unsigned long long>(tag) << 32));
      st_relaxed_u64(P.ylog + it.drow, __float_as_uint(c) | (static_cast<unsigned long long>(tag) << 32));
    }
    const float s2 = it.s2;
    if (it.first) {
      mp = mq = -kInf;
      sp = sq = 0.f;
    }
    {
      const float cm = tile_accumulate<BF16, NV>(wp, s2, tid, nvec, mp, sp);
      if constexpr (CAND) {
        if (it.sketch) store_chunk_max(cm, it.trow, it.t);
      }
    }
    if (pair) {
      load_tile<BF16, NV>(wp, tma, sbase + half, static_cast<const char *>(P.draft) + it.dsrc, tid, nvec,
                          it.len);
    }
    // this warp is done with the stage
    const bool warp_to = __any_sync(FULL_MASK, timed_out);
    __syncwarp();
    if (lane == 0) {
      if (warp_to) ctl.broken = 1;
      mbar_arrive(&ctl.empty[s]);
    }
    if (warp_to) run_to = F_TIMEOUT;
    if (pair) {
      const float cm = tile_accumulate<BF16, NV>(wp, s2, tid, nvec, mq, sq);
      if constexpr (CAND) {
        if (it.sketch && P.drift_m == 0) store_chunk_max(cm, it.drow, it.t);  // (DRIFT: targets only)
      }
    }

    if (it.last && SV_INB(runs % (2 * S), 2 * kMaxStages)) {  // the run ends: fold the CTA's partials
      join_generation();
      const int slot = runs % (2 * S);
      ++runs;
      float Mpw, Spw, Mqw, Sqw;
      fold_max_sum(mp, sp, s2, &Mpw, &Spw);
      fold_max_sum(mq, sq, s2, &Mqw, &Sqw);
      int last = 0;
      if (lane == 0) {
        ctl.wpart[slot][warp] = make_float4(Mpw, Spw, Mqw, Sqw);
        if (run_to) atomicOr(&ctl.tflags[slot], run_to);
        __threadfence_block();
        last = atomicAdd(&ctl.arrived[slot], 1) == NW - 1;
      }
      run_to = 0;
      if (__shfl_sync(FULL_MASK, last, 0)) {
        __threadfence_block();
        const float4 v = lane < NW ? ctl.wpart[slot][lane] : make_float4(-kInf, 0.f, -kInf, 0.f);
        float M1, S1, M2, S2;
        fold_max_sum(v.x, v.y, s2, &M1, &S1);
        fold_max_sum(v.z, v.w, s2, &M2, &S2);
        const uint32_t tf = ctl.tflags[slot];
        SoftPart *rp = P.part + (size_t)it.trow * nt;
        SoftPart *rq = pair ? P.part + (size_t)it.drow * nt : nullptr;
        for (int t = it.run0 + 1 + lane; t <= it.t; t += 32) {
          store_part(rp + t, -kInf, 0.f, 0u, tag);
          if (pair) store_part(rq + t, -kInf, 0.f, 0u, tag);
        }
        if (lane == 0) {
          store_part(rp + it.run0, M1, S1, tf, tag);
          if (pair) store_part(rq + it.run0, M2, S2, tf, tag);
          ctl.arrived[slot] = 0;
          ctl.tflags[slot] = 0;
        }
      }
    }
  }
}

// ============================================================ kernel 2

struct alignas(16) ResolveCtrl {
  float4 mailbox[2];         // this CTA's mass for the cluster exchange
  float wsum[kResolveThreads / 32];
  float Mp, Sp, Mq, Sq;      // normalisers of the stopping position
  float u;                   // its u_sample
  int stop;                  // first rejecting position (K: none)
  uint32_t flags;            // row status bits
  int trunc;                 // the row is truncated (top-k / top-p)
  uint32_t thp, thq;         // key thresholds of the stopping position's p and q
  int klen;                  // entries of the kept list of p at the stopping position (0: none)
  int pad2;
};

// Non-zero ranks copy Mp .. thq (three 16-byte blocks) from rank 0.
static_assert(offsetof(ResolveCtrl, Mp) % 16 == 0 && offsetof(ResolveCtrl, thq) < offsetof(ResolveCtrl, Mp) + 48,
              "the decision fields must be three aligned 16-byte blocks");

// Order-preserving key of a logit value held in fp32 (exact for bf16 logits).
__device__ __forceinline__ uint32_t key_of(float l, bool bf16) {
  const uint32_t u = __float_as_uint(l);
  if (bf16) {
    const uint32_t h = u >> 16;
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  }
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Fold the tile partials of every logit row of row b (target rows 0..K, then
// draft rows 0..K-1) in one round trip: lanes form groups of GS (a power of
// two >= the tile count, at most 32), one group per logit row; lane l of a
// group folds tiles l, l+GS, ... in order, then the group folds in a fixed
// butterfly order.  rstat[r] = (max, sum, draft-token logit, flags).
__device__ bool fold_rows(const ChainStochParams &P, int b, float s2, uint32_t tag, int warp,
                          int lane, float4 *rstat, bool trunc) {
  bool ready = true;  // every record this lane read carries the tag
  constexpr int NW = kResolveThreads / 32;
  const int K = P.K, npos = K + 1, nt = P.nslices;
  int GS = 1;
  while (GS < nt && GS < 32) GS <<= 1;
  const int per_warp = 32 / GS;
  const int sub = lane % GS;
  for (int r0 = warp * per_warp; r0 < npos + K; r0 += NW * per_warp) {
    const int r = r0 + lane / GS;
    float m = -kInf, sacc = 0.f, yv = 0.f;
    uint32_t f = 0;
    if (r < npos + K) {
      const bool draft = r > K;
      const int j = draft ? r - npos : r;
      const int prow = draft ? P.B * npos + b * K + j : b * npos + j;
      if (sub == 0 && trunc && SV_INB(prow, (long long)P.B * (npos + K))) {  // the row's truncation record
        float th, kp;
        uint32_t tf;
        ready &= load_part(P.trunc + prow, tag, &th, &kp, &tf);
      }
      if (sub == 0 && j < K) {
        // the draft token's logit: written only when the token is in range
        const int y = P.tokens && SV_INB((long long)b * K + j, (long long)P.B * K)
                          ? __ldg(P.tokens + (size_t)b * K + j) : -1;
        if (y >= 0 && y < P.V && SV_INB(prow, (long long)P.B * (npos + K))) {
          const unsigned long long w = ld_relaxed_u64(P.ylog + prow);
          yv = __uint_as_float(static_cast<uint32_t>(w));
          ready &= static_cast<uint32_t>(w >> 32) == tag;
        }
      }
      for (int t = sub; t < nt; t += GS) {
        float qm, qs;
        uint32_t qf;
        if (!SV_INB((long long)prow * nt + t, (long long)P.B * (npos + K) * nt)) continue;
        ready &= load_part(P.part + (size_t)prow * nt + t, tag, &qm, &qs, &qf);
        f |= qf;
        const float mn = fmax_nan(m, qm);
        sacc = (m == -kInf ? 0.f : sacc * ex2(__fmul_rn(m - mn, s2))) +
               (qm == -kInf ? 0.f : qs * ex2(__fmul_rn(qm - mn, s2)));
        m = mn;
      }
    }
    // butterfly inside the group
    float M = m;
    for (int o = GS >> 1; o > 0; o >>= 1) M = fmax_nan(M, __shfl_xor_sync(FULL_MASK, M, o));
    float v = (m == -kInf || sacc == 0.f) ? 0.f : sacc * ex2(__fmul_rn(m - M, s2));
    for (int o = GS >> 1; o > 0; o >>= 1) {
      v += __shfl_xor_sync(FULL_MASK, v, o);
      f |= __shfl_xor_sync(FULL_MASK, f, o);
    }
    if (sub == 0 && r < npos + K && SV_INB(r, npos + K)) rstat[r] = make_float4(M, v, yv, __uint_as_float(f));
  }
  return ready;
}

// One row's decisions from the folded statistics: validates the row's inputs,
// forms each ratio in log2 space, finds the first rejection.  One warp; in
// CTA 0 it also writes the diagnostics.
// The scalars lane j of warp 0 needs for position j (first chunk of 32),
// loaded before the dependency wait: they are inputs, never written by the
// stream kernel.
struct RowScalars {
  float us, ua;
  int y;
};

__device__ __forceinline__ RowScalars load_scalars(const ChainStochParams &P, int b, int j) {
  RowScalars r = {0.f, 0.f, -1};
  const int K = P.K;
  if (j <= K && SV_INB((long long)b * (K + 1) + j, (long long)P.B * (K + 1)))
    r.us = __ldg(P.u_sample + (size_t)b * (K + 1) + j);
  if (j < K && SV_INB((long long)b * K + j, (long long)P.B * K)) {
    r.y = __ldg(P.tokens + (size_t)b * K + j);
    r.ua = __ldg(P.u_accept + (size_t)b * K + j);
  }
  return r;
}

__device__ void decide_row(const ChainStochParams &P, int b, float s2, uint32_t tflags, int lane,
                           bool diag, const float4 *rstat, RowScalars first, ResolveCtrl &ctl,
                           bool bf16) {
  const int K = P.K, npos = K + 1, V = P.V;
  uint32_t flags = tflags;
  int tk_;
  float tp_;
  const bool trunc = P.trunc && trunc_active(P, b, V, &tk_, &tp_);
  int stop = K;
  for (int j0 = 0; j0 < npos; j0 += 32) {
    const int j = j0 + lane;
    bool rejects = false;
    float4 tp = make_float4(-kInf, 0.f, 0.f, 0.f), dq = make_float4(-kInf, 0.f, 0.f, 0.f);
    float us = 0.f;
    uint32_t thp = 0, thq = 0;  // truncation thresholds (0: keep all)
    int klen = 0;               // p's kept list (truncated rows)
    if (j < npos) {
      const RowScalars sc = j0 == 0 ? first : load_scalars(P, b, j);
      us = sc.us;
      if (!(us >= 0.f && us < 1.f)) flags |= F_BAD_UNIFORM;
      tp = rstat[j];
      flags |= __float_as_uint(tp.w);
      if (trunc && SV_INB((long long)b * npos + j, (long long)P.B * (npos + K))) {
        // the kept mass replaces the full sum (records already checked)
        float th, kp;
        uint32_t tf;
        load_part(P.trunc + (size_t)b * npos + j, 0u, &th, &kp, &tf);
        flags |= (tf & 1u) ? F_TIMEOUT : 0u;  // bits 1..7: the kept list's length
        thp = __float_as_uint(th);
        klen = static_cast<int>(tf >> 1);
        tp.y = kp;
      }
      if (tp.x != tp.x || tp.x == kInf) flags |= F_NONFINITE;
      else if (tp.x == -kInf) flags |= F_EMPTY;
      if (j < K) {
        const int y = sc.y;
        const float ua = sc.ua;
        if (!(ua >= 0.f && ua < 1.f)) flags |= F_BAD_UNIFORM;
        if (y < 0 || y >= V) flags |= F_BAD_TOKEN;
        dq = rstat[npos + j];
        flags |= __float_as_uint(dq.w);
        if (trunc && SV_INB((long long)P.B * npos + (long long)b * K + j, (long long)P.B * (npos + K))) {
          float th, kp;
          uint32_t tf;
          load_part(P.trunc + (size_t)P.B * npos + (size_t)b * K + j, 0u, &th, &kp, &tf);
          flags |= (tf & 1u) ? F_TIMEOUT : 0u;
          thq = __float_as_uint(th);
          dq.y = kp;
        }
        if (dq.x != dq.x || dq.x == kInf) flags |= F_NONFINITE;
        else if (dq.x == -kInf) flags |= F_EMPTY;
        // ratio p(y)/q(y) in log2 space: identical logits give exactly 0
        // (a token outside a truncated law has probability 0)
        const float l2p = key_of(tp.z, bf16) < thp ? -kInf
                        : __fadd_rn(__fmaf_rn(tp.z, s2, -__fmul_rn(tp.x, s2)), -lg2(tp.y));
        const float l2q = key_of(dq.z, bf16) < thq ? -kInf
                        : __fadd_rn(__fmaf_rn(dq.z, s2, -__fmul_rn(dq.x, s2)), -lg2(dq.y));
        const float l2r = __fadd_rn(l2p, -l2q);
        rejects = !((l2r >= 0.f) || (ua < ex2(l2r)));
        if (diag && SV_INB((long long)b * K + j, (long long)P.B * K)) {
          const size_t d = (size_t)b * K + j;
          if (P.p_at_draft) P.p_at_draft[d] = ex2(l2p);
          if (P.q_at_draft) P.q_at_draft[d] = ex2(l2q);
        }
      }
    }
    const unsigned rej = __ballot_sync(FULL_MASK, rejects);
    const bool found_here = stop == K && rej;
    const int src = found_here ? __ffs(rej) - 1 : K - j0;  // stop lane, or the bonus lane
    if ((found_here || (stop == K && j0 + 32 >= npos)) && lane == src) {
      ctl.Mp = tp.x;
      ctl.Sp = tp.y;
      ctl.Mq = found_here ? dq.x : -kInf;
      ctl.Sq = found_here ? dq.y : 0.f;
      ctl.u = us;
      ctl.thp = thp;
      ctl.thq = found_here ? thq : 0u;
      ctl.klen = klen;
    }
    if (found_here) stop = j0 + src;
  }
  flags = __reduce_or_sync(FULL_MASK, flags);
  if (diag && P.resid_mass)
    for (int j = lane; j < K; j += 32)
      if (j != stop && SV_INB((long long)b * K + j, (long long)P.B * K)) P.resid_mass[(size_t)b * K + j] = 0.f;
  if (lane == 0) {
    ctl.stop = stop;
    ctl.flags = flags;
    ctl.trunc = trunc;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kResolveThreads, kResolveBlocksPerSm) chain_resolve_kernel(const __grid_constant__ ChainStochParams P) {
  using F = Fmt<BF16>;
  constexpr int NT = kResolveThreads, NW = NT / 32, EPV = F::EPV, ESZ = F::ESZ;
  __shared__ ResolveCtrl ctl;
  extern __shared__ __align__(16) unsigned char rsm[];
  float4 *rstat = reinterpret_cast<float4 *>(rsm);                         // [2K+1]
  float *rsum = reinterpret_cast<float *>(rsm + (size_t)(2 * P.K + 1) * 16);  // [rounds][NT]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int crank = (int)cluster_ctarank(), C = (int)cluster_nctarank();
  const int b = (int)cluster_id_x();
  const int K = P.K, npos = K + 1, V = P.V;
  const float T = P.temperature ? __ldg(P.temperature + b) : 1.0f;
  const uint32_t tflags = (T > 0.f && T < kInf) ? 0u : F_BAD_TEMPERATURE;
  const float s2 = tflags ? 1.f : __fdiv_rn(kLog2e, T);
  // The next call's generation step may launch once every CTA of this grid
  // runs: it waits, resident, for this grid to complete before it advances
  // the tag.
  allow_dependents();

  // The logits are inputs the kernel before this one (the stream, or the
  // truncation kernel) never writes, so the rows where walks most often stop
  // (position 0) can be pulled into L2 before waiting.
  if (tid == 0 && P.use_tma) {
    const int s0p = crank * P.L;
    const int lenp = max(0, min(V, s0p + P.L) - s0p);
    if (lenp > 0) {
      bulk_prefetch_l2(static_cast<const char *>(P.target) + ((size_t)(b * npos) * V + s0p) * ESZ,
                       static_cast<uint32_t>(lenp) * ESZ);
      if (K > 0)
        bulk_prefetch_l2(static_cast<const char *>(P.draft) + ((size_t)(b * K) * V + s0p) * ESZ,
                         static_cast<uint32_t>(lenp) * ESZ);
    }
  }
  // Block 0 waits for the kernel before this one on its way out, so this
  // grid never completes before the one it depends on.
  auto join_stream = [&]() {
    if (blockIdx.x == 0 && tid == 0) grid_dependency_wait();
  };
  // Every CTA of the cluster polls the row's partial records (and, when
  // truncated, its truncation records) until every one carries this call's
  // tag -- the kernel before this one stamps them as it goes, so a row is
  // resolved as soon as its own records are in, not when that whole grid is
  // done -- folds them and takes the walk's decisions itself: the same
  // arithmetic in the same order gives the same bits in every CTA, so the
  // draw starts without a cluster barrier.  The CTAs agree on the row's
  // status at the draw's one barrier (a wait that gave up in one CTA only
  // flags the row there).
  {
    const RowScalars first = load_scalars(P, b, lane);
    const uint32_t tag = *reinterpret_cast<volatile const uint32_t *>(P.gen);
    // a truncated verify also polls the row's truncation records, stamped
    // the same way, so rows resolve while the truncation grid still runs
    int tk_;
    float tp_;
    const bool trunc = P.trunc && trunc_active(P, b, V, &tk_, &tp_);
    bool gave_up = false;
    const uint64_t t0 = global_timer_ns();
    while (!__syncthreads_and(fold_rows(P, b, s2, tag, warp, lane, rstat, trunc))) {
      if (__syncthreads_or(global_timer_ns() - t0 > P.wait_limit_ns)) {  // bounded
        gave_up = true;
        break;
      }
      __nanosleep(200);
    }
    if (warp == 0)
      decide_row(P, b, s2, tflags | (gave_up ? F_TIMEOUT : 0u), lane, crank == 0, rstat, first, ctl, BF16);
    __syncthreads();
  }
  const uint32_t my_flags = ctl.flags;
  const int stop = ctl.stop;

  const float nMp = -__fmul_rn(ctl.Mp, s2), nMq = -__fmul_rn(ctl.Mq, s2);
  const float iSp = __frcp_rn(ctl.Sp), iSq = ctl.Sq > 0.f ? __frcp_rn(ctl.Sq) : 0.f;
  const float u = ctl.u;
  const float2 s2v = make_float2(s2, s2), nMpv = make_float2(nMp, nMp), nMqv = make_float2(nMq, nMq);
  const float2 iSpv = make_float2(iSp, iSp), niSqv = make_float2(-iSq, -iSq);
  const int s0 = crank * P.L;
  const int len = [&] {
    const int l = max(0, min(V, s0 + P.L) - s0);
    // bounds build: the stopping position's slice of this CTA must lie in
    // the logit tensors, else the CTA reads nothing (the row comes out wrong)
    if (!(SV_INB(b, P.B) && SV_INB(stop, npos) &&
          SV_INR((long long)(b * npos + stop) * V + s0, l, (long long)P.B * npos * V) &&
          (stop == K || SV_INR((long long)(b * K + stop) * V + s0, l, (long long)P.B * K * V))))
      return 0;
    return l;
  }();
  const int nr = P.vpw / 32;  // rounds of 32 vectors per warp
  const int vbase = warp * P.vpw;
  const bool aligned = P.use_tma != 0;
  const char *tg = static_cast<const char *>(P.target) + ((size_t)(b * npos + stop) * V + s0) * ESZ;
  const char *dg = stop < K
                       ? static_cast<const char *>(P.draft) + ((size_t)(b * K + stop) * V + s0) * ESZ
                       : nullptr;

  int task = stop < K ? 1 : 2;  // 1: residual [p - q]+, 2: the target law p
  uint32_t row_flags = 0;       // every CTA's status bits, from the exchange
  float Z = 0.f;
  int xs = 0;
  int owner_cta = -1;
  float t_c = 0.f;
  // mass of element e of a vector pair under the current task (with
  // truncation, tokens below a law's threshold have probability 0)
  const bool trunc = ctl.trunc != 0;
  const uint32_t thp = ctl.thp, thq = ctl.thq;
  auto mass = [&](const uint32_t *wp, const uint32_t *wq, int e) {
    const bool kp = !trunc || order_key<BF16>(elem_bits<BF16>(wp, e)) >= thp;
    const float pe = kp ? ex2(__fmaf_rn(F::elem(wp, e), s2, nMp)) : 0.f;
    if (task == 2) return pe;
    const bool kq = !trunc || order_key<BF16>(elem_bits<BF16>(wq, e)) >= thq;
    const float qe = kq ? ex2(__fmaf_rn(F::elem(wq, e), s2, nMq)) : 0.f;
    return fmaxf(__fmaf_rn(pe, iSp, -__fmul_rn(qe, iSq)), 0.f);
  };
  // A truncated row whose kept set of p at the stopping position came as a
  // list with its record draws from that list: p, and so the residual, is 0
  // outside it, and nothing else of the row is read.  The CTAs agree on it
  // at the exchange, as on the row's status.
  const bool by_list = trunc && ctl.klen > 0;
  bool list_draw = false;
  while (true) {
    // ---- pass: per-round masses (kept for the search), then the CTA total
    float tsum = 0.f;
    if (by_list) {
      // no pass: the list is drawn from after the exchange
    } else if (trunc) {
      // truncated laws: four rounds of target loads in flight, then element
      // by element with the thresholds -- only where some element of the
      // target vector may reach p's threshold (the draft vector is loaded
      // just then): elsewhere p' is 0 and so is the vector's mass under
      // either task, exactly
      const float thp_f = key_value<BF16>(thp);
      const uint32_t thp_w = pack_threshold<BF16>(thp_f);
#pragma unroll 1
      for (int k0 = 0; k0 < nr; k0 += 4) {
        uint32_t wp[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int vlen = (k0 + k < nr) ? len : 0;  // rounds past nr read nothing
          F::load_vec(wp[k], nullptr, tg, aligned, vbase + 32 * (k0 + k) + lane, vlen);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float r = 0.f;
          if (may_reach_bits<BF16>(wp[k], thp_w, thp_f) != 0) {
            uint32_t wq[4];
            if (task == 1) {
              const int vlen = (k0 + k < nr) ? len : 0;
              F::load_vec(wq, nullptr, dg, aligned, vbase + 32 * (k0 + k) + lane, vlen);
            }
#pragma unroll
            for (int e = 0; e < EPV; ++e) r += mass(wp[k], wq, e);
          }
          if (k0 + k < nr) rsum[(k0 + k) * NT + tid] = r;
          tsum += r;
        }
      }
    } else if (aligned && task == 1) {
#pragma unroll 1
      for (int k0 = 0; k0 < nr; k0 += 4) {
        uint4 vp[4], vq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int v = vbase + 32 * (k0 + k) + lane;
          const bool in = (k0 + k < nr) && v * EPV < len;
          vp[k] = in ? __ldg(reinterpret_cast<const uint4 *>(tg) + v) : make_uint4(F::NEG_INF_WORD, F::NEG_INF_WORD, F::NEG_INF_WORD, F::NEG_INF_WORD);
          vq[k] = in ? __ldg(reinterpret_cast<const uint4 *>(dg) + v) : make_uint4(F::NEG_INF_WORD, F::NEG_INF_WORD, F::NEG_INF_WORD, F::NEG_INF_WORD);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t *wp = reinterpret_cast<const uint32_t *>(&vp[k]);
          const uint32_t *wq = reinterpret_cast<const uint32_t *>(&vq[k]);
          // element pairs through packed fp32: the same per-element values
          // as mass(); only the order of the vector's sum differs
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < EPV / 2; ++i) {
            const float2 ap = ffma2(F::pair(wp, i), s2v, nMpv);
            const float2 aq = ffma2(F::pair(wq, i), s2v, nMqv);
            const float2 t = fmul2(make_float2(ex2(aq.x), ex2(aq.y)), niSqv);
            const float2 d = ffma2(make_float2(ex2(ap.x), ex2(ap.y)), iSpv, t);
            acc = fadd2(acc, make_float2(fmaxf(d.x, 0.f), fmaxf(d.y, 0.f)));
          }
          const float r = acc.x + acc.y;
          if (k0 + k < nr) rsum[(k0 + k) * NT + tid] = r;
          tsum += r;
        }
      }
    } else if (aligned) {
#pragma unroll 1
      for (int k0 = 0; k0 < nr; k0 += 4) {
        uint4 vp[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int v = vbase + 32 * (k0 + k) + lane;
          const bool in = (k0 + k < nr) && v * EPV < len;
          vp[k] = in ? __ldg(reinterpret_cast<const uint4 *>(tg) + v) : make_uint4(F::NEG_INF_WORD, F::NEG_INF_WORD, F::NEG_INF_WORD, F::NEG_INF_WORD);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t *wp = reinterpret_cast<const uint32_t *>(&vp[k]);
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < EPV / 2; ++i) {
            const float2 ap = ffma2(F::pair(wp, i), s2v, nMpv);
            acc = fadd2(acc, make_float2(ex2(ap.x), ex2(ap.y)));
          }
          const float r = acc.x + acc.y;
          if (k0 + k < nr) rsum[(k0 + k) * NT + tid] = r;
          tsum += r;
        }
      }
    } else {  // rows that are not 16-byte aligned: element loads with masking
#pragma unroll 1
      for (int k0 = 0; k0 < nr; k0 += 4) {
        uint32_t wp[4][4], wq[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int v = vbase + 32 * (k0 + k) + lane;
          const int vlen = (k0 + k < nr) ? len : 0;  // rounds past nr read nothing
          F::load_vec(wp[k], nullptr, tg, false, v, vlen);
          if (task == 1) F::load_vec(wq[k], nullptr, dg, false, v, vlen);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float r = 0.f;
#pragma unroll
          for (int e = 0; e < EPV; ++e) r += mass(wp[k], wq[k], e);
          if (k0 + k < nr) rsum[(k0 + k) * NT + tid] = r;
          tsum += r;
        }
      }
    }
    const float wsum = warp_sum(tsum);
    if (lane == 0) ctl.wsum[warp] = wsum;
    __syncthreads();
    if (tid == 0) {
      float c = 0.f;
      for (int w2 = 0; w2 < NW; ++w2) c += ctl.wsum[w2];
      ctl.mailbox[xs] = make_float4(c, __uint_as_float(my_flags), by_list ? 1.f : 0.f, 0.f);
    }
    cluster_sync();
    const float4 mb = lane < C ? ld_dsmem_f4(dsmem_addr(&ctl.mailbox[xs], (uint32_t)lane))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    const float cm = mb.x;
    xs ^= 1;
    row_flags = __reduce_or_sync(FULL_MASK, __float_as_uint(mb.y));
    if (row_flags) break;  // the row's status: no token
    const int n_list = static_cast<int>(__reduce_add_sync(FULL_MASK, lane < C && mb.z != 0.f ? 1u : 0u));
    if (n_list != 0) {  // (the same records give every CTA the same choice)
      if (n_list == C) list_draw = true;
      else row_flags = F_TIMEOUT;
      break;
    }
    const float tot = sum_lanes(cm, C);
    if (task == 1 && !(tot > 0.f)) {  // the residual vanished in fp32: draw from p
      task = 2;
      continue;
    }
    if (task == 1) Z = tot;
    owner_cta = pick_entry(cm, C, u * tot, &t_c);
    break;
  }
  cluster_arrive();  // done with the peers' mailboxes

  // the row's outputs, by one warp
  auto write_row = [&](int token) {
    for (int j = lane; j < npos && SV_INB(b, P.B); j += 32) {
      const int o = j < stop ? __ldg(P.tokens + (size_t)b * K + j) : (j == stop ? token : -1);
      P.out_tokens[(size_t)b * npos + j] = o;
    }
    if (lane == 0 && SV_INB(b, P.B)) {
      P.accepted_len[b] = stop;
      P.num_emitted[b] = stop + 1;
      P.row_status[b] = 0;
      if (stop < K && P.resid_mass) P.resid_mass[(size_t)b * K + stop] = Z;
    }
  };
  if (row_flags) {  // the agreed status: rank 0 writes the row's outputs
    if (crank == 0 && warp == 0 && SV_INB(b, P.B)) {
      for (int j = lane; j < npos; j += 32) P.out_tokens[(size_t)b * npos + j] = -1;
      if (lane == 0) {
        P.accepted_len[b] = -1;
        P.num_emitted[b] = 0;
        P.row_status[b] = lowest_code(row_flags);
      }
    }
  } else if (list_draw) {
    // Rank 0's warp 0 draws from the kept list of p at the stopping position
    // (at most 64 entries, key desc): the masses under the task, in vocabulary
    // order, then the first entry whose cumulative mass exceeds u times the
    // total, or the last one with mass.
    if (crank == 0 && warp == 0) {
      __threadfence();  // the list was written before the record polled above
      const int n = min(ctl.klen, kKeptMax);
      const int prow = b * npos + stop;
      const unsigned long long *kl = P.klist + (size_t)prow * kKeptMax;
      int tok[2];
      float pe[2], ms[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        const bool in = i < n && SV_INB((long long)prow * kKeptMax + i, (long long)P.B * npos * kKeptMax);
        const unsigned long long ent = in ? ld_relaxed_u64(kl + i) : 0ull;
        tok[h] = in ? static_cast<int>(~static_cast<uint32_t>(ent)) : 0x7fffffff;
        const float lp = key_value<BF16>(static_cast<uint32_t>(ent >> 32));
        pe[h] = in ? ex2(__fmaf_rn(lp, s2, nMp)) : 0.f;
        ms[h] = pe[h];
        if (in && task == 1 && SV_INB(tok[h], V)) {
          const size_t at = ((size_t)b * K + stop) * V + tok[h];
          uint32_t bits;
          if constexpr (BF16) bits = __ldg(static_cast<const unsigned short *>(P.draft) + at);
          else bits = __ldg(static_cast<const unsigned int *>(P.draft) + at);
          const float ld = BF16 ? __uint_as_float(bits << 16) : __uint_as_float(bits);
          const float qe = order_key<BF16>(bits) >= thq ? ex2(__fmaf_rn(ld, s2, nMq)) : 0.f;
          ms[h] = fmaxf(__fmaf_rn(pe[h], iSp, -__fmul_rn(qe, iSq)), 0.f);
        }
      }
      // vocabulary order: each entry's rank among the token ids
      int rk[2] = {0, 0};
      for (int j2 = 0; j2 < n; ++j2) {
        const int tj = __shfl_sync(FULL_MASK, j2 < 32 ? tok[0] : tok[1], j2 & 31);
        rk[0] += tj < tok[0] ? 1 : 0;
        rk[1] += tj < tok[1] ? 1 : 0;
      }
      float *s_ms = rsum, *s_pe = rsum + kKeptMax;
      int *s_tok = reinterpret_cast<int *>(rsum + 2 * kKeptMax);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (lane + 32 * h < n) {
          s_ms[rk[h]] = ms[h];
          s_pe[rk[h]] = pe[h];
          s_tok[rk[h]] = tok[h];
        }
      }
      __syncwarp();
      auto scan = [&](const float *src, float &m0, float &m1, float &c0, float &c1) {
        m0 = lane < n ? src[lane] : 0.f;
        m1 = lane + 32 < n ? src[lane + 32] : 0.f;
        c0 = warp_inclusive_scan(m0, lane);
        c1 = warp_inclusive_scan(m1, lane) + __shfl_sync(FULL_MASK, c0, 31);
      };
      float m0, m1, c0, c1;
      scan(s_ms, m0, m1, c0, c1);
      float tot = __shfl_sync(FULL_MASK, c1, 31);
      if (task == 1 && tot > 0.f) Z = tot;
      if (task == 1 && !(tot > 0.f)) {  // the residual vanished in fp32: draw from p
        task = 2;
        scan(s_pe, m0, m1, c0, c1);
        tot = __shfl_sync(FULL_MASK, c1, 31);
      }
      const float t = __fmul_rn(ctl.u, tot);
      const unsigned h0 = __ballot_sync(FULL_MASK, m0 > 0.f && c0 > t);
      const unsigned h1 = __ballot_sync(FULL_MASK, m1 > 0.f && c1 > t);
      int pos;
      if (h0) pos = __ffs(h0) - 1;
      else if (h1) pos = 31 + __ffs(h1);
      else {  // past the total: the last entry with mass
        const unsigned p0 = __ballot_sync(FULL_MASK, m0 > 0.f), p1 = __ballot_sync(FULL_MASK, m1 > 0.f);
        pos = p1 ? 63 - __clz(p1) : (p0 ? 31 - __clz(p0) : 0);
      }
      write_row(s_tok[pos]);
    }
  } else if (crank == owner_cta) {
    float t_w;
    const float wm = lane < NW ? ctl.wsum[lane] : 0.f;
    const int owner_warp = pick_entry(wm, NW, t_c, &t_w);
    if (warp == owner_warp) {
      // round of 32 vectors, then lane, then element, in vocabulary order
      int ks = -1, klast = -1;
      float t1 = 0.f, acc = 0.f;
      for (int k = 0; k < nr; ++k) {
        const float Wk = warp_sum(rsum[k * NT + tid]);
        const float prev = acc;
        acc += Wk;
        if (Wk > 0.f) {
          klast = k;
          if (ks < 0 && acc > t_w) {
            ks = k;
            t1 = t_w - prev;
          }
        }
      }
      if (ks < 0) {
        ks = klast;
        t1 = kInf;
      }
      int token = -1;
      if (ks >= 0) {
        const float my = rsum[ks * NT + tid];
        const int v = vbase + 32 * ks + lane;
        uint32_t wp[4], wq[4];
        F::load_vec(wp, nullptr, tg, aligned, v, len);
        if (task == 1) F::load_vec(wq, nullptr, dg, aligned, v, len);
        const float incl = warp_inclusive_scan(my, lane);
        float excl = __shfl_up_sync(FULL_MASK, incl, 1);
        if (lane == 0) excl = 0.f;
        const unsigned hit = __ballot_sync(FULL_MASK, my > 0.f && incl > t1);
        int ls;
        bool clamp = false;
        if (hit) {
          ls = __ffs(hit) - 1;
        } else {
          ls = 31 - __clz(__ballot_sync(FULL_MASK, my > 0.f));
          clamp = true;
        }
        int pos = -1;
        if (lane == ls) {
          const float t3 = clamp ? kInf : t1 - excl;
          float c = 0.f;
          int es = -1, elast = -1;
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float m = mass(wp, wq, e);
            c += m;
            if (m > 0.f) {
              elast = e;
              if (es < 0 && c > t3) es = e;
            }
          }
          if (es < 0) es = elast;
          pos = s0 + v * EPV + es;
        }
        token = __shfl_sync(FULL_MASK, pos, ls);
      }
      write_row(token);
    }
  }
  cluster_wait();  // no CTA leaves while a peer may still read its mailbox
  join_stream();
}

// ============================================================ block selection
//
// Block-wide radix selection, 8 bits a pass from the top, of the r-th
// largest key of a set that `each(f)` enumerates (every thread hands its own
// keys to f).  Needs at least r keys.  Returns the key; n_above and n_equal
// count the keys above it and equal to it.  Every thread of the block calls
// it; chist (256 ints), s_digit and s_above are shared scratch.
template <int KEYBITS, int NT, typename Each>
__device__ uint32_t block_kth_largest(Each each, int r, int *chist, int *s_digit, int *s_above,
                                      int &n_above, int &n_equal) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, pmask = 0;
  int rem = r, in = 0;
  for (int shift = KEYBITS - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) chist[i] = 0;
    __syncthreads();
    each([&](uint32_t k) {
      if ((k & pmask) == prefix) atomicAdd(&chist[(k >> shift) & 255u], 1);
    });
    __syncthreads();
    if (warp == 0) {  // lane l owns bins 255-8l .. 248-8l
      int cnt[8], own = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = chist[255 - 8 * lane - i];
        own += cnt[i];
      }
      int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += n;
      }
      int above = incl - own;
      if (above < rem && rem <= incl) {
        int dgt = 255 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above + cnt[i] >= rem) {
            dgt = 255 - 8 * lane - i;
            break;
          }
          above += cnt[i];
        }
        *s_digit = dgt;
        *s_above = above;
      }
    }
    __syncthreads();
    const int dgt = *s_digit;
    rem -= *s_above;
    in = chist[dgt];
    prefix |= static_cast<uint32_t>(dgt) << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  n_above = r - rem;
  n_equal = in;
  return prefix;
}

// ============================================================ DRIFT
//
// "Speculative Decoding Under Distribution Shift: DRIFT Recalibration" (the
// residual paragraph of its method): at every drafted position, restrict
// target and draft to the m tokens of highest target probability and report
// log p - log q there.  The ring stream reads positions 0 .. K-1 of target
// and draft (records for both, chunk maxima for the target rows); then
// drift_pick_kernel (one CTA per position j < K of row b, with the
// truncation kernels below) takes the m largest target keys from the chunks
// those maxima point to, equal keys at the boundary in vocabulary order, so
// the support matches the oracle's exactly; drift_finish_kernel forms the
// residuals.

constexpr int kDriftFinishThreads = 256;
constexpr int kDriftMaxM = kDriftMaxSupport;

constexpr int kDriftCand = 2048;  // candidate list of the sampled-threshold path
constexpr int kDriftSample = 64;  // sampling stride of that threshold, in vectors

// Elements of a V-long row in its sampled vectors (every kDriftSample-th
// vector of EPV elements, the last one possibly short).
__device__ __forceinline__ int sampled_count(int V, int epv) {
  const int nvec = (V + epv - 1) / epv;
  const int last = ((nvec - 1) / kDriftSample) * kDriftSample;  // last sampled vector
  return (last / kDriftSample) * epv + min(epv, V - last * epv);
}

// A row's (max, sum) from its slices' (max, sum) pairs, in one fixed order:
// lane t folds slices t, t + 32, ... in order, then the lanes fold in a fixed
// butterfly (fold_max_sum).  slice(t, &m, &s) returns false for a record that
// is not in yet; the result is whether every lane's were.
template <typename Slice>
__device__ __forceinline__ bool fold_slice_stats(int nt, int lane, float s2, Slice slice, float *M,
                                                 float *S) {
  float mm = -kInf, ss = 0.f;
  bool ready = true;
  for (int t = lane; t < nt; t += 32) {
    float qm, qs;
    ready &= slice(t, &qm, &qs);
    const float mn = fmax_nan(mm, qm);
    ss = (mm == -kInf ? 0.f : ss * ex2(__fmul_rn(mm - mn, s2))) +
         (qm == -kInf ? 0.f : qs * ex2(__fmul_rn(qm - mn, s2)));
    mm = mn;
  }
  fold_max_sum(mm, ss, s2, M, S);
  return __all_sync(FULL_MASK, ready);
}

// DRIFT, last kernel: one CTA per row, a programmatic dependent of the pick
// grid (which completes only after the stream grid has), so both grids'
// writes are visible after its dependency wait.  The row status ORs every
// position's flags from the pick kernel's records (a record that did not
// come is a timeout); a flagged row gets support -1 and residual NaN
// everywhere, since no single pick CTA sees the whole row.
template <bool BF16>
__global__ void __launch_bounds__(kDriftFinishThreads) drift_finish_kernel(const __grid_constant__ ChainStochParams P) {
  __shared__ uint32_t row_f;
  grid_dependency_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K = P.K, m = P.drift_m;
  const uint32_t tag = *reinterpret_cast<volatile const uint32_t *>(P.gen);
  if (tid == 0) row_f = 0u;
  __syncthreads();
  for (int j = tid; j < K && SV_INB(j, kDriftMaxK); j += kDriftFinishThreads) {
    float M1, S1;
    uint32_t f1 = 0;
    const bool in = load_part(P.trunc_area + (size_t)b * K + j, tag, &M1, &S1, &f1);
    const uint32_t f = in ? f1 : F_TIMEOUT;
    if (f) atomicOr(&row_f, f);
  }
  __syncthreads();
  const uint32_t f = row_f;
  if (tid == 0 && P.row_status) P.row_status[b] = lowest_code(f);
  if (f) {
    int32_t *sup = P.drift_support + (size_t)b * K * m;
    float *res = P.drift_residual + (size_t)b * K * m;
    for (int i = tid; i < K * m; i += kDriftFinishThreads) {
      sup[i] = -1;
      res[i] = __int_as_float(0x7fc00000);
    }
  }
}

// Largest key x (0 .. 2^bits - 1) with pred(x) true, pred being monotone
// (true for small x).
template <typename Pred>
__device__ __forceinline__ uint32_t largest_key(int bits, Pred pred) {
  uint32_t x = 0;
  for (int bit = bits - 1; bit >= 0; --bit) {
    const uint32_t c = x | (1u << bit);
    if (pred(c)) x = c;
  }
  return x;
}

// ============================================================ truncation
//
// "Speculative Decoding: Draft, Verify, and Correct", 'Preserve the
// distribution you actually intend': when top-k / top-p define the sampling
// law, acceptance and correction use the truncated p, and q is the truncated
// law that produced the draft.  Per logit row the selection kernel finds the
// key threshold theta of the kept set -- top-k: the largest theta with at
// least k keys >= theta (boundary ties kept); then top-p: the largest theta
// whose keys >= theta carry at least top_p of the top-k mass -- and the kept
// mass.  Sums run in a fixed order, so the result is deterministic.
//
// The ring stream (CAND) leaves, for every truncated logit row, the maximum
// of each consumer thread's chunk of every tile.  The k-th largest chunk
// maximum is at most the row's k-th largest logit (k chunks hold a logit at
// least that large), so every logit the top-k keeps lies in a chunk whose
// maximum reaches it: the selection re-reads only those chunks (about k of
// c3's 4096) and takes their logits at or above it as candidates.  A row
// whose candidates cannot settle the thresholds (too many chunks or
// candidates, or a nucleus that reaches below them) takes a sampled
// threshold and lists its candidates in a pass over its own logits, and
// after that searches the whole row.

// The sample rank r of a row's sampled threshold: about r * kDriftSample of
// its keys reach the r-th largest sampled key.
__device__ __forceinline__ int trunc_sample_rank(int tk) {
  return tk > 0 ? max(16, (2 * tk) / kDriftSample + 2) : 16;
}

// The selection CTA: 192 threads, six per SM (c3's 704 logit rows in one
// wave; 56 registers, none spilled -- at 256 threads and five per SM the
// kernel spilled, and its warp sort ran 7 times slower).
constexpr int kSelThreads = 192;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxRowTiles = (SPEC_MAX_V + kSoftMinSlice - 1) / kSoftMinSlice;
constexpr int kMaxRowChunks = kMaxRowTiles * kSoftThreads;
constexpr int kMaxSelChunks = 256;  // chunks one row re-reads at most
constexpr int kTopPChunks = 64;     // chunks a top-p-only row starts from

// The r-th largest of n 16-bit keys in shared memory (n even, 1 <= r <= n),
// bit by bit from the top: the largest th with at least r keys >= th.  Each
// step is one block-wide count; red holds two rounds of per-warp counts.
// Every thread of the block calls it.
template <int NT>
__device__ uint32_t kth_largest_key16(const unsigned short *keys, int n, int r, int (*red)[NT / 32]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t *wk = reinterpret_cast<const uint32_t *>(keys);
  const int nw = n / 2;
  uint32_t th = 0;
#pragma unroll 1
  for (int bit = 15; bit >= 0; --bit) {
    const uint32_t c = th | (1u << bit);
    int cnt = 0;
    for (int w = tid; w < nw; w += NT) {
      const uint32_t x = wk[w];
      cnt += ((x & 0xFFFFu) >= c ? 1 : 0) + ((x >> 16) >= c ? 1 : 0);
    }
    cnt = __reduce_add_sync(FULL_MASK, cnt);
    int *slot = red[bit & 1];
    if (lane == 0) slot[warp] = cnt;
    __syncthreads();
    int tot = 0;
#pragma unroll
    for (int w2 = 0; w2 < NT / 32; ++w2) tot += slot[w2];
    if (tot >= r) th = c;
  }
  return th;
}

// Scratch of chunk_candidates, kept in the calling kernel's control block.
struct ChunkScratch {
  int clist[kMaxSelChunks];  // chunks to re-read
  uint32_t aux[kSelThreads]; // the threads' largest keys, then the keys above their bound
  int cred[2][kSelWarps];    // counts of the threshold search
  int n_surv, n_chunks, n_cand;
  uint32_t bound;
};

// The candidates of one logit row from its chunk maxima (nch of them in
// shared memory, the top 16 bits of each chunk's largest order key): the
// rc-th largest maximum th is the threshold, and every logit of a chunk whose
// maximum reaches th is listed into ck as (key << 32) | ~index when its key
// reaches th too.  Every logit of the row whose key reaches th is listed.
// ck may share memory with the maxima (they are read before it is written).
// With exact false, th is the lower bound below instead (also at most the
// row's rc-th largest logit: fewer steps, a few more candidates).  Returns
// the candidate count (possibly above cap, which ck holds at most), or -1
// when more than kMaxSelChunks chunks reach th.  The 192 threads of the
// block call it.
template <bool BF16>
__device__ int chunk_candidates(const unsigned short *chunk, int nch, int rc, const char *src,
                                bool aligned, int nvec, int V, ChunkScratch &cs,
                                unsigned long long *ck, int cap, bool exact) {
  using F = Fmt<BF16>;
  constexpr int EPV = F::EPV;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    cs.n_chunks = 0;
    cs.n_cand = 0;
  }
  // A lower bound first: the rc-th largest of the threads' largest keys (rc
  // threads hold a key at least that large, so at least rc keys reach it);
  // only the keys that reach it can be th, and warp 0 searches those when
  // they are few.
  const uint32_t *wk = reinterpret_cast<const uint32_t *>(chunk);
  const int nw = nch / 2;
  auto warp_kth = [&](int n) {  // warp 0: the rc-th largest of aux[0 .. n), n <= kSelThreads
    constexpr int PL = kSelThreads / 32;
    uint32_t v[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) v[i] = lane + 32 * i < n ? cs.aux[lane + 32 * i] : 0u;
    uint32_t x = 0;
#pragma unroll 1
    for (int bit = 15; bit >= 0; --bit) {  // (a candidate is >= 1: padding never counts)
      const uint32_t c = x | (1u << bit);
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < PL; ++i) cnt += v[i] >= c ? 1 : 0;
      if (static_cast<int>(__reduce_add_sync(FULL_MASK, static_cast<unsigned>(cnt))) >= rc) x = c;
    }
    return x;
  };
  {
    uint32_t tmax = 0;
    for (int w = tid; w < nw; w += kSelThreads) {
      const uint32_t x = wk[w];
      tmax = max(tmax, max(x & 0xFFFFu, x >> 16));
    }
    cs.aux[tid] = tmax;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t lb = warp_kth(kSelThreads);
    if (lane == 0) {
      cs.bound = lb;
      cs.n_surv = 0;
    }
  }
  __syncthreads();
  if (exact) {
    const uint32_t lb = cs.bound;
    for (int w = tid; w < nw; w += kSelThreads) {
      const uint32_t x = wk[w];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t k = h ? (x >> 16) : (x & 0xFFFFu);
        if (k >= lb) {
          const int slot = atomicAdd(&cs.n_surv, 1);
          if (slot < kSelThreads) cs.aux[slot] = k;
        }
      }
    }
  }
  uint32_t th = cs.bound;
  if (exact) {
    __syncthreads();
    if (cs.n_surv <= kSelThreads) {
      if (warp == 0) {
        const uint32_t x = warp_kth(cs.n_surv);
        if (lane == 0) cs.bound = x;
      }
      __syncthreads();
      th = cs.bound;
    } else {
      th = kth_largest_key16<kSelThreads>(chunk, nch, rc, cs.cred);
    }
  }
  // the chunks whose maximum reaches it
  for (int c = tid; c < nch; c += kSelThreads) {
    if (chunk[c] >= th) {
      const int slot = atomicAdd(&cs.n_chunks, 1);
      if (slot < kMaxSelChunks) cs.clist[slot] = c;
    }
  }
  __syncthreads();
  const int nsel = cs.n_chunks;
  if (nsel > kMaxSelChunks) return -1;
  // their vectors, all loads in flight at once, then every logit whose key
  // reaches th (the maxima keep the top 16 bits of a logit's key)
  constexpr int PERV = (kMaxSelChunks * kSoftVecs + kSelThreads - 1) / kSelThreads;
  uint32_t w[PERV][4];
  int vid[PERV];
#pragma unroll
  for (int q2 = 0; q2 < PERV; ++q2) {
    const int i = tid + q2 * kSelThreads;  // (chunk i / kSoftVecs, vector i % kSoftVecs)
    vid[q2] = -1;
    if (i < nsel * kSoftVecs) {
      const int c = cs.clist[i / kSoftVecs];
      const int t = c / kSoftThreads, lt = c - t * kSoftThreads;
      vid[q2] = t * (kSoftThreads * kSoftVecs) + lt + (i % kSoftVecs) * kSoftThreads;
    }
    F::load_vec(w[q2], nullptr, src, aligned, vid[q2] < 0 ? nvec : vid[q2], V);
  }
  __syncthreads();  // the maxima are read: the candidates may overwrite them
#pragma unroll
  for (int q2 = 0; q2 < PERV; ++q2) {
    if (vid[q2] < 0) continue;
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const uint32_t bits = elem_bits<BF16>(w[q2], e);
      const uint32_t k = order_key<BF16>(bits);
      const uint32_t k16 = BF16 ? k : (k >> 16);
      const int idx = vid[q2] * EPV + e;
      if (k16 >= th && idx < V) {
        const int slot = atomicAdd(&cs.n_cand, 1);
        if (slot < cap) ck[slot] = (static_cast<unsigned long long>(k) << 32) | (~static_cast<uint32_t>(idx));
      }
    }
  }
  __syncthreads();
  return cs.n_cand;
}

struct alignas(16) TruncCtrl {
  // the row's chunk maxima, then (once they are used) the candidates:
  // (key << 32) | (~token id), which sorts key desc, id asc, and their
  // masses, then prefix sums
  union {
    unsigned short chunk[kMaxRowChunks];
    struct {
      unsigned long long ck[kDriftCand];
      float e[kDriftCand];
    };
  };
  ChunkScratch cs;
  int settled;               // warp 0's settling of a small list: 1 done, 0 retry
  uint32_t theta_w;
  float kept_w;
  int kept_n;                // entries of the kept set (a prefix of the sorted list)
  float fred[kSelWarps];
  int ired[kSelWarps];
  int chist[256];
  int n_cand, digit, above, pos;
  float M, S;
  uint32_t flags;
};

template <bool BF16>
__global__ void __launch_bounds__(kSelThreads, 6) trunc_select_kernel(const __grid_constant__ ChainStochParams P) {
  using F = Fmt<BF16>;
  constexpr int EPV = F::EPV, ESZ = F::ESZ;
  constexpr int KEYBITS = BF16 ? 16 : 32;
  __shared__ TruncCtrl ctl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = P.K, V = P.V, npos = K + 1, nt = P.nslices;
  // CTAs in batch-row order (row b's target positions, then its drafts), so
  // rows complete one after another and the resolve kernel, which polls each
  // row's records, finishes most rows while this grid still runs.
  const int b = blockIdx.x / (npos + K), q = blockIdx.x - b * (npos + K);
  const bool is_target = q < npos;
  const int j = is_target ? q : q - npos;
  const int row = is_target ? b * npos + j : P.B * npos + b * K + j;
  // The stream has completed, and with it the generation step: its tile
  // records and chunk maxima are in, and the tag read below is this call's.
  grid_dependency_wait();
  allow_dependents();
  // forced-timeout test: no record of this call appears, so the resolve
  // kernel's bounded wait gives up
  if (P.force_timeout) return;
  int tk;
  float tp;
  if (!trunc_active(P, b, V, &tk, &tp)) return;
  float T = P.temperature ? __ldg(P.temperature + b) : 1.0f;
  if (!(T > 0.f && T < kInf)) T = 1.0f;  // the resolve kernel flags the row
  const float s2 = __fdiv_rn(kLog2e, T);
  const uint32_t tag = *reinterpret_cast<volatile const uint32_t *>(P.gen);
  const char *src = static_cast<const char *>(is_target ? P.target : P.draft) + (size_t)row_offset(P, row) * ESZ;
  const bool aligned = P.use_tma != 0;
  const int nvec = (V + EPV - 1) / EPV;
  auto bits_at = [&](int i) -> uint32_t {
    if constexpr (BF16) return __ldg(reinterpret_cast<const unsigned short *>(src) + i);
    else return __ldg(reinterpret_cast<const unsigned int *>(src) + i);
  };
  // block sums in a fixed order
  auto block_sum_i = [&](int v) {
    v = __reduce_add_sync(FULL_MASK, v);
    if (lane == 0) ctl.ired[warp] = v;
    __syncthreads();
    int t = 0;
    for (int w2 = 0; w2 < kSelWarps; ++w2) t += ctl.ired[w2];
    __syncthreads();
    return t;
  };
  auto block_sum_f = [&](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
    if (lane == 0) ctl.fred[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w2 = 0; w2 < kSelWarps; ++w2) t += ctl.fred[w2];
    __syncthreads();
    return t;
  };
  // The chunk maxima a row starts from: rc of them, the row's top_k, or
  // kTopPChunks for top-p alone.  Their copy into shared memory starts now
  // and lands while warp 0 folds the records.
  const int nch = nt * kSoftThreads;
  const int rc = tk > 0 ? tk : min(kTopPChunks, nch);
  const bool use_chunks = rc <= kMaxSelChunks && rc <= nch && nch <= kMaxRowChunks;
  if (use_chunks) {
    const uint4 *srcm = reinterpret_cast<const uint4 *>(P.cmax + (size_t)row * nch);
    const int nv = nch / 8;  // every row's maxima start 512-byte aligned
    for (int v = tid; v < nv; v += kSelThreads)
      if (SV_INB((long long)row * nv + v, (long long)P.B * (2 * K + 1) * nv))
        cp_async16(reinterpret_cast<uint4 *>(ctl.chunk) + v, srcm + v);
  }
  // The row's tile records (lane t of warp 0: tiles t and t + 32), loaded
  // now and folded once the candidates are gathered.
  unsigned long long rec_a[2] = {0ull, 0ull}, rec_b[2] = {0ull, 0ull};
  if (warp == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = lane + 32 * h;
      if (t < nt && SV_INB((long long)row * nt + t, (long long)P.B * (2 * K + 1) * nt)) {
        rec_a[h] = ld_relaxed_u64(&P.part[(size_t)row * nt + t].a);
        rec_b[h] = ld_relaxed_u64(&P.part[(size_t)row * nt + t].b);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  SoftPart *rec = P.trunc + row;
  float nM = 0.f;  // -M s2, once the records are folded
  auto mass_of = [&](uint32_t bits) {  // exp2((l - M) s2) of one element
    const float l = BF16 ? __uint_as_float(bits << 16) : __uint_as_float(bits);
    return l == -kInf ? 0.f : ex2(__fmaf_rn(l, s2, nM));
  };
  // ---- sampled thresholds, for rows the chunks cannot settle: the r-th
  // largest of the keys of every kDriftSample-th vector
  constexpr int kNSV = (SPEC_MAX_V + EPV * kDriftSample * kSelThreads - 1) / (EPV * kDriftSample * kSelThreads);
  const int n_samples = sampled_count(V, EPV);
  auto sample_tau = [&](int r) -> uint32_t {
    if (r > n_samples) return 0u;
    uint32_t smp[kNSV][4];
#pragma unroll
    for (int q2 = 0; q2 < kNSV; ++q2)
      F::load_vec(smp[q2], nullptr, src, aligned, (tid + q2 * kSelThreads) * kDriftSample, V);
    auto samples = [&](auto f) {
#pragma unroll
      for (int q2 = 0; q2 < kNSV; ++q2) {
        const int v = (tid + q2 * kSelThreads) * kDriftSample;
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          if (v * EPV + e < V) f(order_key<BF16>(elem_bits<BF16>(smp[q2], e)));
      }
    };
    int na, ne;
    return block_kth_largest<KEYBITS, kSelThreads>(samples, r, ctl.chist, &ctl.digit, &ctl.above, na, ne);
  };
  // ---- one pass over the row listing every key >= tau (a lane visits only
  // its elements not below tau and appends them one by one: they are sorted
  // later).  Returns the candidate count.
  auto pass = [&](uint32_t tau) {
    if (tid == 0) ctl.n_cand = 0;
    const float tau_f = key_value<BF16>(tau);
    const uint32_t tau_w = pack_threshold<BF16>(tau_f);
    __syncthreads();
    constexpr int U = 2;
    for (int v00 = tid; v00 < nvec; v00 += 2 * U * kSelThreads) {
      uint32_t wab[2][U][4];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int u = 0; u < U; ++u)
          F::load_vec(wab[h][u], nullptr, src, aligned, v00 + (h * U + u) * kSelThreads, V);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int v0 = v00 + h * U * kSelThreads;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          uint32_t msk = may_reach_bits<BF16>(wab[h][u], tau_w, tau_f);
          while (msk) {
            const int e = __ffs(msk) - 1;
            msk &= msk - 1;
            const int idx = (v0 + u * kSelThreads) * EPV + e;
            const uint32_t k = order_key<BF16>(elem_bits_at<BF16>(wab[h][u], e));
            if (k >= tau && idx < V) {
              const int slot = atomicAdd(&ctl.n_cand, 1);
              if (slot < kDriftCand)
                ctl.ck[slot] = (static_cast<unsigned long long>(k) << 32) | (~static_cast<uint32_t>(idx));
            }
          }
        }
      }
    }
    __syncthreads();
    return ctl.n_cand;
  };
  // the listed candidates' masses, from their keys, once M is known
  auto fill_masses = [&](int n) {
    for (int i = tid; i < min(n, kDriftCand); i += kSelThreads) {
      const float l = key_value<BF16>(static_cast<uint32_t>(ctl.ck[i] >> 32));
      ctl.e[i] = l == -kInf ? 0.f : ex2(__fmaf_rn(l, s2, nM));
    }
    __syncthreads();
  };
  auto key_at = [&](int i) { return static_cast<uint32_t>(ctl.ck[i] >> 32); };
  // ---- sort the candidates (key desc, id asc) and prefix-sum their masses
  auto sort_and_scan = [&](int nc) {
    int N = 64;
    while (N < nc) N <<= 1;
    for (int i = nc + tid; i < N; i += kSelThreads) {
      ctl.ck[i] = 0ull;
      ctl.e[i] = 0.f;
    }
    __syncthreads();
    for (int size = 2; size <= N; size <<= 1) {  // bitonic, descending
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int t = tid; t < N / 2; t += kSelThreads) {
          const int lo = 2 * t - (t & (stride - 1)), hi = lo + stride;
          const bool up = (lo & size) == 0;
          const unsigned long long a = ctl.ck[lo], c = ctl.ck[hi];
          if ((a < c) == up) {
            ctl.ck[lo] = c;
            ctl.ck[hi] = a;
            const float t0 = ctl.e[lo];
            ctl.e[lo] = ctl.e[hi];
            ctl.e[hi] = t0;
          }
        }
        __syncthreads();
      }
    }
    // inclusive prefix sums in sorted order: PER consecutive per thread
    constexpr int PER = (kDriftCand + kSelThreads - 1) / kSelThreads;
    float v[PER], run = 0.f;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int i = tid * PER + q;
      run += i < N ? ctl.e[i] : 0.f;
      v[q] = run;
    }
    float incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) ctl.fred[warp] = incl;
    __syncthreads();
    float off = incl - run;
    for (int w2 = 0; w2 < warp; ++w2) off += ctl.fred[w2];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int i = tid * PER + q;
      if (i < N) ctl.e[i] = off + v[q];
    }
    __syncthreads();
  };
  // The same sort and scan for sets of at most 64 (a top-k set, normally):
  // warp 0 holds entry i = lane + 32 h in registers and runs the same bitonic
  // network with shuffles (the keys are unique but for the zero padding), so
  // no block barrier is needed until it writes the 64 entries back.
  auto warp_sort_and_scan = [&](int nc) {
    if (warp == 0) {
      unsigned long long k[2];
      float e[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        k[h] = i < nc ? ctl.ck[i] : 0ull;
        e[h] = i < nc ? ctl.e[i] : 0.f;
      }
#pragma unroll
      for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          if (stride == 32) {  // entries lane (lower) and lane + 32, ascending block: up
            if (k[0] < k[1]) {
              const unsigned long long tk0 = k[0];
              k[0] = k[1];
              k[1] = tk0;
              const float te0 = e[0];
              e[0] = e[1];
              e[1] = te0;
            }
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int i = lane + 32 * h;
              const bool lower = (i & stride) == 0, up = (i & size) == 0;
              const unsigned long long pk = __shfl_xor_sync(FULL_MASK, k[h], stride);
              const float pe = __shfl_xor_sync(FULL_MASK, e[h], stride);
              // the pair swaps when (lower's key < upper's key) == up
              if ((lower ? (k[h] < pk) : (pk < k[h])) == up) {
                k[h] = pk;
                e[h] = pe;
              }
            }
          }
        }
      }
      // inclusive prefix sums in sorted order
      float s0 = e[0], s1 = e[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float n0 = __shfl_up_sync(FULL_MASK, s0, o), n1 = __shfl_up_sync(FULL_MASK, s1, o);
        if (lane >= o) {
          s0 += n0;
          s1 += n1;
        }
      }
      s1 += __shfl_sync(FULL_MASK, s0, 31);
      ctl.ck[lane] = k[0];
      ctl.ck[lane + 32] = k[1];
      ctl.e[lane] = s0;
      ctl.e[lane + 32] = s1;
    }
    __syncthreads();
  };
  // A list of at most 64 candidates, settled without a sorting network:
  // thread i < n takes candidate i's mass and its rank (the candidates whose
  // (key, ~id) is larger: the keys are unique) and puts both at that rank,
  // which is the order of warp_sort_and_scan; warp 0 then forms its prefix
  // sums and the boundaries of the code below (the k-th key's group of ties;
  // the first prefix that reaches top_p of the kept mass, and its group) by
  // ballots.  The same arithmetic in the same order gives the same threshold
  // and kept mass.
  //
  // A list of up to kSelThreads candidates under top-k is settled the same
  // way from its 64 highest: the kept set lies among them unless the k-th
  // key's group of ties reaches rank 63 (settled = 2: the block path below
  // takes the list).
  auto settle_small = [&](int n_all) {
    const int n = min(n_all, 64);
    unsigned long long *sk = ctl.ck + kDriftCand / 2;  // the 64 highest, sorted
    if (tid < n_all) {
      const unsigned long long mine = ctl.ck[tid];
      int rank = 0;
#pragma unroll 4
      for (int j2 = 0; j2 < n_all; ++j2) rank += ctl.ck[j2] > mine ? 1 : 0;
      if (rank < 64) {
        const float l = key_value<BF16>(static_cast<uint32_t>(mine >> 32));
        sk[rank] = mine;
        ctl.e[rank] = l == -kInf ? 0.f : ex2(__fmaf_rn(l, s2, nM));
      }
    }
    __syncthreads();
    if (warp != 0) return;
    unsigned long long k[2];
    float e[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      k[h] = i < n ? sk[i] : 0ull;
      e[h] = i < n ? ctl.e[i] : 0.f;
    }
    float s0 = e[0], s1 = e[1];
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      const float n0 = __shfl_up_sync(FULL_MASK, s0, o), n1 = __shfl_up_sync(FULL_MASK, s1, o);
      if (lane >= o) {
        s0 += n0;
        s1 += n1;
      }
    }
    s1 += __shfl_sync(FULL_MASK, s0, 31);
    const uint32_t k0 = static_cast<uint32_t>(k[0] >> 32), k1 = static_cast<uint32_t>(k[1] >> 32);
    auto key_at_w = [&](int i) {  // sorted entry i's key (every lane gets it)
      const uint32_t a0 = __shfl_sync(FULL_MASK, k0, i & 31), a1 = __shfl_sync(FULL_MASK, k1, i & 31);
      return i < 32 ? a0 : a1;
    };
    auto prefix_at_w = [&](int i) {
      const float a0 = __shfl_sync(FULL_MASK, s0, i & 31), a1 = __shfl_sync(FULL_MASK, s1, i & 31);
      return i < 32 ? a0 : a1;
    };
    auto group_end = [&](int i) {  // last entry (< n) with entry i's key
      const uint32_t ki = key_at_w(i);
      const unsigned b0 = __ballot_sync(FULL_MASK, lane < n && k0 == ki);
      const unsigned b1 = __ballot_sync(FULL_MASK, lane + 32 < n && k1 == ki);
      return b1 ? 63 - __clz(b1) : 31 - __clz(b0);
    };
    if (n_all > n && (tk > n || group_end(tk - 1) == n - 1)) {  // the kept set may go past rank 63
      if (lane == 0) ctl.settled = 2;
      return;
    }
    int gk = n - 1;
    float Sk = ctl.S;
    if (tk > 0) {
      gk = group_end(tk - 1);
      Sk = prefix_at_w(gk);
    }
    int ok = 1, kn = 0;
    uint32_t th = 0;
    float kp = 0.f;
    if (tp < 1.f) {
      const float target = __fmul_rn(tp, Sk);
      if (tk == 0 && !(prefix_at_w(n - 1) >= target)) {
        ok = 0;
      } else {
        const unsigned c0 = __ballot_sync(FULL_MASK, lane <= gk && s0 >= target);
        const unsigned c1 = __ballot_sync(FULL_MASK, lane + 32 <= gk && s1 >= target);
        const int pos = c0 ? __ffs(c0) - 1 : (c1 ? 31 + __ffs(c1) : gk);
        const int ge = group_end(pos);
        th = key_at_w(pos);
        kp = prefix_at_w(ge);
        kn = ge + 1;
      }
    } else {
      th = key_at_w(gk);
      kp = Sk;
      kn = gk + 1;
    }
    if (lane == 0) {
      ctl.settled = ok;
      ctl.theta_w = th;
      ctl.kept_w = kp;
      ctl.kept_n = kn;
    }
  };
  uint32_t theta = 0;
  float kept = 0.f;
  int klen = 0;  // entries of the kept list written for the resolve kernel
  bool done = false;
  int r = trunc_sample_rank(tk);
  // the candidates from the chunk maxima (-1: they cannot give a list)
  int nc = use_chunks ? chunk_candidates<BF16>(ctl.chunk, nch, rc, src, aligned, nvec, V, ctl.cs, ctl.ck, kDriftCand,
                                               tk == 0)
                      : -1;
  // ---- the row's max and sum from the stream's tile records (warp 0); a
  // record missing or flagged, or a non-finite or empty row, gets no
  // thresholds (the resolve kernel reports the row from the same records)
  if (warp == 0) {
    float Mw, Sw;
    uint32_t f = 0;
    const bool ready = fold_slice_stats(nt, lane, s2, [&](int t, float *m, float *s) {
      uint32_t qf = 0;
      const int h = t >> 5;  // t = lane + 32 h
      const bool ok = decode_part(h ? rec_a[1] : rec_a[0], h ? rec_b[1] : rec_b[0], tag, m, s, &qf);
      f |= qf;
      return ok;
    }, &Mw, &Sw);
    f = __reduce_or_sync(FULL_MASK, f);
    if (lane == 0) {
      ctl.M = Mw;
      ctl.S = Sw;
      ctl.flags = (!ready || f || Mw != Mw || Mw == kInf || Mw == -kInf) ? 1u : 0u;
    }
  }
  __syncthreads();
  if (ctl.flags) {
    if (tid == 0) store_part(rec, 0.f, 0.f, 1u, tag);
    return;
  }
  nM = -__fmul_rn(ctl.M, s2);
  // attempt 0 takes the chunks' candidates; 1 to 3 a sampled threshold each
  for (int attempt = nc >= 0 ? 0 : 1; attempt < 4 && !done; ++attempt) {
    if (attempt > 0) nc = pass(sample_tau(r));
    if (nc > kDriftCand) {  // too many: raise the threshold
      if (r <= 1) break;
      r = max(1, r / 4);
      continue;
    }
    if (nc < max(tk, 1)) {  // the top k are not all candidates: lower it
      r *= 4;
      continue;
    }
    bool small_done = false;
    if (nc <= 64 || (tk > 0 && nc <= kSelThreads)) {  // a small list: ranks, then warp 0
      settle_small(nc);
      __syncthreads();
      const int st = ctl.settled;
      __syncthreads();
      if (st == 0) {  // (top-p alone) the nucleus reaches below the list
        r *= 4;
        continue;
      }
      small_done = st == 1;
    }
    if (small_done) {
      theta = ctl.theta_w;
      kept = ctl.kept_w;
      // a target row's kept set, in the order above, for the resolve kernel
      // (its record, stored after this, gives the length)
      if (is_target) {
        const int kn = ctl.kept_n;
        if (tid < kn && SV_INB((long long)row * kKeptMax + tid, (long long)P.B * npos * kKeptMax)) {
          P.klist[(size_t)row * kKeptMax + tid] = ctl.ck[kDriftCand / 2 + tid];
          __threadfence();
        }
        klen = kn;
      }
      __syncthreads();
      done = true;
      break;
    }
    fill_masses(nc);
    // With top-k only the candidates at or above the k-th largest key (ties
    // included) can be kept, and the nucleus lies among them: select that key
    // by radix, keep those candidates, sort only them.  Their order and prefix
    // sums are those of the full sort's first entries, so a set of 64 or
    // fewer goes to the warp sort whole.
    int ns = nc;
    if (tk > 0 && nc > 64) {
      auto cand_keys = [&](auto f) {
        for (int i = tid; i < nc; i += kSelThreads) f(key_at(i));
      };
      int na, ne;
      const uint32_t thk = block_kth_largest<KEYBITS, kSelThreads>(cand_keys, tk, ctl.chist, &ctl.digit,
                                                                    &ctl.above, na, ne);
      constexpr int PER = (kDriftCand + kSelThreads - 1) / kSelThreads;
      unsigned long long kk[PER];
      float ee[PER];
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int i = tid + q * kSelThreads;
        kk[q] = i < nc ? ctl.ck[i] : 0ull;
        ee[q] = i < nc ? ctl.e[i] : 0.f;
      }
      if (tid == 0) ctl.n_cand = 0;
      __syncthreads();
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int i = tid + q * kSelThreads;
        if (i < nc && static_cast<uint32_t>(kk[q] >> 32) >= thk) {
          const int slot = atomicAdd(&ctl.n_cand, 1);
          ctl.ck[slot] = kk[q];
          ctl.e[slot] = ee[q];
        }
      }
      __syncthreads();
      ns = ctl.n_cand;
    }
    if (ns <= 64) warp_sort_and_scan(ns);
    else sort_and_scan(ns);
    // top-k: the k-th candidate's key, through the end of its group of ties
    int gk = ns - 1;
    float Sk = ctl.S;
    if (tk > 0) {
      if (tid == 0) {
        int g = tk - 1;
        while (g + 1 < ns && key_at(g + 1) == key_at(tk - 1)) ++g;
        ctl.pos = g;
      }
      __syncthreads();
      gk = ctl.pos;
      Sk = ctl.e[gk];
    }
    if (tp < 1.f) {
      const float target = __fmul_rn(tp, Sk);
      if (tk == 0 && !(ctl.e[ns - 1] >= target)) {  // the nucleus reaches below tau
        r *= 4;
        __syncthreads();
        continue;
      }
      if (tid == 0) {  // first prefix reaching the target, then the end of its group
        int lo = 0, hi = gk;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (ctl.e[mid] >= target) hi = mid;
          else lo = mid + 1;
        }
        int g = lo;
        while (g + 1 < ns && key_at(g + 1) == key_at(lo)) ++g;
        ctl.pos = lo;
        ctl.digit = g;
      }
      __syncthreads();
      theta = key_at(ctl.pos);
      kept = ctl.e[ctl.digit];
    } else {
      theta = key_at(gk);
      kept = Sk;
    }
    done = true;
  }
  if (!done) {
    // the whole row: the same searches, every evaluation one pass over it
    auto row_count = [&](uint32_t x) {
      int c = 0;
      for (int i = tid; i < V; i += kSelThreads) c += order_key<BF16>(bits_at(i)) >= x;
      return block_sum_i(c);
    };
    auto row_mass = [&](uint32_t x) {
      float sm = 0.f;
      for (int i = tid; i < V; i += kSelThreads) {
        const uint32_t bits = bits_at(i);
        if (order_key<BF16>(bits) >= x) sm += mass_of(bits);
      }
      return block_sum_f(sm);
    };
    uint32_t thk = 0;
    float Sk = ctl.S;
    if (tk > 0) {
      thk = largest_key(KEYBITS, [&](uint32_t x) { return row_count(x) >= tk; });
      Sk = row_mass(thk);
    }
    if (tp < 1.f) {
      const float target = __fmul_rn(tp, Sk);
      theta = largest_key(KEYBITS, [&](uint32_t x) { return row_mass(x) >= target; });
      kept = row_mass(theta);
    } else {
      theta = thk;
      kept = Sk;
    }
  }
  // flags bits 1..7: the kept list's length (at most 64)
  if (tid == 0) store_part(rec, __uint_as_float(theta), kept, static_cast<uint32_t>(klen) << 1, tag);
}

// ---- DRIFT's pick: one CTA of kSelThreads per drafted position j < K of
// row b, a programmatic dependent of the ring stream (no bonus position;
// chunk maxima for the target rows).

constexpr int kPickCand = kSelThreads;  // candidates ranked one per thread

struct alignas(16) PickCtrl {
  // the row's chunk maxima, then (once they are used) the candidates, or
  // the whole-row radix histograms of the fallback
  union {
    unsigned short chunk[kMaxRowChunks];
    unsigned long long ck[kPickCand];
    int hist[kSelWarps][256];
  };
  ChunkScratch cs;
  int sel_idx[kDriftMaxM];
  uint32_t sel_key[kDriftMaxM];
  int scan[kSelWarps];
  int n_gt, n_eq, digit, above;
  float Mp, Sp;     // the target row's max and sum
  float Mq, lSq;    // the draft row's max and log2 sum
  uint32_t tflags, dflags, flags;
};

template <bool BF16>
__global__ void __launch_bounds__(kSelThreads, 6) drift_pick_kernel(const __grid_constant__ ChainStochParams P) {
  using F = Fmt<BF16>;
  constexpr int EPV = F::EPV, ESZ = F::ESZ;
  constexpr int KEYBITS = BF16 ? 16 : 32;
  constexpr int NW = kSelWarps;
  __shared__ PickCtrl ctl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = P.K, npos = K + 1, V = P.V, m = P.drift_m, nt = P.nslices;
  const int b = blockIdx.x / K, j = blockIdx.x - b * K;
  const int row = b * npos + j;  // the target row of position j
  // The stream has completed, and with it the generation step: its tile
  // records and chunk maxima are in, and the tag read below is this call's.
  grid_dependency_wait();
  allow_dependents();
  // forced-timeout test: no record of this call appears, so the finishing
  // kernel reports a timeout
  if (P.force_timeout) return;
  const float T = P.temperature ? __ldg(P.temperature + b) : 1.0f;
  const uint32_t tflags = (T > 0.f && T < kInf) ? 0u : F_BAD_TEMPERATURE;
  const float s2 = __fdiv_rn(kLog2e, tflags ? 1.0f : T);  // the stream's (a bad T flags the row)
  const uint32_t tag = *reinterpret_cast<volatile const uint32_t *>(P.gen);
  int32_t *sup = P.drift_support + ((size_t)b * K + j) * m;
  float *res = P.drift_residual + ((size_t)b * K + j) * m;
  const char *tg = static_cast<const char *>(P.target) + (size_t)row * V * ESZ;
  const bool aligned = P.use_tma != 0;
  const int nvec = (V + EPV - 1) / EPV;
  // the chunk maxima (copied while warp 0 loads the tile records)
  const int nch = nt * kSoftThreads;
  const bool use_chunks = m <= kMaxSelChunks && m <= nch && nch <= kMaxRowChunks;
  if (use_chunks) {
    const uint4 *srcm = reinterpret_cast<const uint4 *>(P.cmax + (size_t)row * nch);
    const int nv = nch / 8;
    for (int v = tid; v < nv; v += kSelThreads)
      if (SV_INB((long long)row * nv + v, (long long)P.B * (2 * K + 1) * nv))
        cp_async16(reinterpret_cast<uint4 *>(ctl.chunk) + v, srcm + v);
  }
  // tile records: warp 0 the target row's, warp 1 the draft row's (the
  // stream's row numbering), folded once the candidates are listed
  const long long drow = (long long)P.B * npos + (long long)b * K + j;
  unsigned long long rec_a[2] = {0ull, 0ull}, rec_b[2] = {0ull, 0ull};
  if (warp <= 1) {
    const long long r = warp == 0 ? row : drow;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = lane + 32 * h;
      if (t < nt && SV_INB(r * nt + t, (long long)P.B * (2 * K + 1) * nt)) {
        rec_a[h] = ld_relaxed_u64(&P.part[(size_t)r * nt + t].a);
        rec_b[h] = ld_relaxed_u64(&P.part[(size_t)r * nt + t].b);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  const int nc = use_chunks ? chunk_candidates<BF16>(ctl.chunk, nch, m, tg, aligned, nvec, V, ctl.cs, ctl.ck, kPickCand,
                                                     false)
                            : -1;
  // ---- the target row's and the draft row's max and sum, each folded from
  // its tile records in one fixed order (identical rows give identical
  // bits); this position's flags go to the finishing kernel in a stamped
  // record
  if (warp <= 1) {
    float M1, S1;
    uint32_t rf = 0;
    const bool ready = fold_slice_stats(nt, lane, s2, [&](int t, float *qm, float *qs) {
      uint32_t qf = 0;
      const int h = t >> 5;  // t = lane + 32 h
      const bool ok = decode_part(h ? rec_a[1] : rec_a[0], h ? rec_b[1] : rec_b[0], tag, qm, qs, &qf);
      rf |= qf;
      return ok;
    }, &M1, &S1);
    rf = __reduce_or_sync(FULL_MASK, rf);
    if (lane == 0) {
      uint32_t f = ready && !rf ? 0u : F_TIMEOUT;
      if (M1 != M1 || M1 == kInf) f |= F_NONFINITE;
      else if (M1 == -kInf) f |= F_EMPTY;
      if (warp == 0) {
        ctl.tflags = f;
        ctl.Mp = M1;
        ctl.Sp = S1;
      } else {
        ctl.dflags = f;
        ctl.Mq = M1;
        ctl.lSq = lg2(S1);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t f = tflags | ctl.tflags | ctl.dflags;
    ctl.flags = f;
    store_part(P.trunc_area + (size_t)b * K + j, ctl.Mp, ctl.Sp, f, tag);
  }
  __syncthreads();
  if (ctl.flags) {  // the finishing kernel blanks the whole row
    for (int i = tid; i < m; i += kSelThreads) {
      sup[i] = -1;
      res[i] = __int_as_float(0x7fc00000);
    }
    return;
  }
  const float nMp = -__fmul_rn(ctl.Mp, s2);
  const float l2Sp = lg2(ctl.Sp);
  const float nMq = -__fmul_rn(ctl.Mq, s2), l2Sq = ctl.lSq;
  // support entry `rank` is token ii with target logit lt: log2 p and log2 q
  // as in the walk, the residual log p - log q in nats (a masked draft logit
  // gives +inf)
  auto emit = [&](int rank, int ii, float lt) {
    const size_t at = ((size_t)b * K + j) * V + ii;
    float ld;
    if constexpr (BF16) ld = bf16_lo(__ldg(static_cast<const unsigned short *>(P.draft) + at));
    else ld = __ldg(static_cast<const float *>(P.draft) + at);
    const float l2p = __fadd_rn(__fmaf_rn(lt, s2, nMp), -l2Sp);
    const float l2q = ld == -kInf ? -kInf : __fadd_rn(__fmaf_rn(ld, s2, nMq), -l2Sq);
    sup[rank] = ii;
    res[rank] = __fmul_rn(__fadd_rn(l2p, -l2q), kLn2);
  };
  if (nc >= m && nc <= kPickCand) {
    // every logit at or above the threshold is a candidate: the m of highest
    // (key, ~id) are the support, in that order
    if (tid < nc) {
      const unsigned long long mine = ctl.ck[tid];
      int rank = 0;
#pragma unroll 4
      for (int q = 0; q < nc; ++q) rank += ctl.ck[q] > mine ? 1 : 0;
      if (rank < m) emit(rank, static_cast<int>(~static_cast<uint32_t>(mine)),
                         key_value<BF16>(static_cast<uint32_t>(mine >> 32)));
    }
    return;
  }
  // ---- fallback (the chunks cannot give the list: ties over too many
  // chunks, or too many candidates): radix selection of the m-th largest
  // key over the whole row, 8 bits a pass from the top
  auto bits_at = [&](int i) -> uint32_t {
    if constexpr (BF16) return __ldg(reinterpret_cast<const unsigned short *>(tg) + i);
    else return __ldg(reinterpret_cast<const unsigned int *>(tg) + i);
  };
  __syncthreads();
  uint32_t prefix = 0, pmask = 0;
  int rem = m;  // rank still to find within the keys matching prefix
  int last_count = 0;
  for (int shift = KEYBITS - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < NW * 256; i += kSelThreads) (&ctl.hist[0][0])[i] = 0;
    __syncthreads();
    for (int v = tid; v < nvec; v += kSelThreads) {
      uint32_t w[4];
      F::load_vec(w, nullptr, tg, aligned, v, V);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const uint32_t k = order_key<BF16>(elem_bits<BF16>(w, e));
        if ((k & pmask) == prefix && v * EPV + e < V) {
          const uint32_t d = (k >> shift) & 255u;
          const unsigned same = __match_any_sync(__activemask(), d);
          if (lane == __ffs(same) - 1) atomicAdd(&ctl.hist[warp][d], __popc(same));
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < 256; i += kSelThreads) {
      int c = 0;
      for (int w2 = 0; w2 < NW; ++w2) c += ctl.hist[w2][i];
      ctl.hist[0][i] = c;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending); suffix counts from the top
      int cnt[8], own = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = ctl.hist[0][255 - 8 * lane - i];
        own += cnt[i];
      }
      int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += n;
      }
      int above = incl - own;  // keys in higher bins than this lane's
      if (above < rem && rem <= incl) {
        int dgt = 255 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above + cnt[i] >= rem) {
            dgt = 255 - 8 * lane - i;
            break;
          }
          above += cnt[i];
        }
        ctl.digit = dgt;
        ctl.above = above;
      }
    }
    __syncthreads();
    const int dgt = ctl.digit;
    rem -= ctl.above;
    last_count = ctl.hist[0][dgt];
    prefix |= static_cast<uint32_t>(dgt) << shift;
    pmask |= 255u << shift;
    __syncthreads();  // hist and digit are reused by the next pass
  }
  const uint32_t tkey = prefix;  // key of the m-th largest
  const int n_gt = m - rem;      // keys above it, all selected
  // ---- collect: every key above tkey; rem keys equal to it, lowest index first
  if (tid == 0) {
    ctl.n_gt = 0;
    ctl.n_eq = 0;
  }
  __syncthreads();
  const bool take_all_eq = last_count == rem;
  for (int v = tid; v < nvec; v += kSelThreads) {
    uint32_t w[4];
    F::load_vec(w, nullptr, tg, aligned, v, V);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const int idx = v * EPV + e;
      if (idx >= V) continue;
      const uint32_t k = order_key<BF16>(elem_bits<BF16>(w, e));
      if (k > tkey) {
        const int slot = atomicAdd(&ctl.n_gt, 1);
        if (SV_INB(slot, kDriftMaxM)) {
          ctl.sel_idx[slot] = idx;
          ctl.sel_key[slot] = k;
        }
      } else if (k == tkey && take_all_eq) {
        const int slot = n_gt + atomicAdd(&ctl.n_eq, 1);
        if (SV_INB(slot, kDriftMaxM)) {
          ctl.sel_idx[slot] = idx;
          ctl.sel_key[slot] = k;
        }
      }
    }
  }
  if (!take_all_eq) {
    // ties straddle the boundary: each thread counts the equal keys of its
    // contiguous index range, an exclusive scan orders them, and the first
    // rem in vocabulary order are taken
    const int span = (V + kSelThreads - 1) / kSelThreads;
    const int i0 = min(V, tid * span), i1 = min(V, i0 + span);
    int mine = 0;
    for (int i = i0; i < i1; ++i) mine += order_key<BF16>(bits_at(i)) == tkey;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) ctl.scan[warp] = incl;
    __syncthreads();
    int base = incl - mine;
    for (int w2 = 0; w2 < warp; ++w2) base += ctl.scan[w2];
    for (int i = i0; i < i1 && base < rem; ++i) {
      if (order_key<BF16>(bits_at(i)) == tkey && SV_INB(n_gt + base, kDriftMaxM)) {
        ctl.sel_idx[n_gt + base] = i;
        ctl.sel_key[n_gt + base] = tkey;
        ++base;
      }
    }
  }
  __syncthreads();
  // ---- rank (key descending, index ascending) among the m selected
  for (int i = tid; i < m; i += kSelThreads) {
    const uint32_t ki = ctl.sel_key[i];
    const int ii = ctl.sel_idx[i];
    int rank = 0;
    for (int q = 0; q < m; ++q) {
      const uint32_t kq = ctl.sel_key[q];
      rank += (kq > ki) || (kq == ki && ctl.sel_idx[q] < ii);
    }
    emit(rank, ii, key_value<BF16>(ki));
  }
}

size_t resolve_smem(const ChainStochParams &p) {
  return static_cast<size_t>(2 * p.K + 1) * 16 + static_cast<size_t>(p.vpw / 32) * kResolveThreads * 4;
}

// The resolve kernel's attributes are set once per device, so steady-state
// launches make no other driver calls and can be captured into a CUDA graph.
// The ring stream kernel's shared-memory attribute, set once per device
// (again only when more is needed).
template <bool BF16, int NV, int S, bool CAND = false>
cudaError_t prepare_ring(size_t smem) {
  static std::atomic<size_t> done_smem[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done_smem[dev].load() >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(softmax_partials_kernel<BF16, NV, S, CAND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e == cudaSuccess) done_smem[dev].store(smem);
  return e;
}

template <bool BF16>
cudaError_t prepare(int cluster) {
  static std::atomic<int> done_nonportable[kMaxDevices];
  static std::atomic<int> done_resolve[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!done_resolve[dev].load()) {
    e = cudaFuncSetAttribute(chain_resolve_kernel<BF16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    done_resolve[dev].store(1);
  }
  if (cluster > 8 && !done_nonportable[dev].load()) {
    e = cudaFuncSetAttribute(chain_resolve_kernel<BF16>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    done_nonportable[dev].store(1);
  }
  return cudaSuccess;
}

// Advances the workspace's generation word (the call's tag) and clears the
// stream's claim counter: one thread, launched as a programmatic dependent of
// the kernel before it, so it is resident and waiting when that kernel ends.
// It lets the stream launch only once that kernel (and so every kernel before
// it, the producers of this call's logits included) has completed: the
// stream reads its inputs from its first instruction on.
__global__ void advance_generation_kernel(uint32_t *gen, uint32_t *claim) {
  grid_dependency_wait();
  allow_dependents();
  // the tag is never 0, so zero-filled memory never passes for a record
  const uint32_t g = *gen + 1u;
  *gen = g ? g : 1u;
  *claim = 0u;
}

// The resolve kernel: a cluster of `cluster` CTAs per row, a programmatic
// dependent of the kernel launched just before it.
template <bool BF16>
cudaError_t launch_resolve(const ChainStochParams &p, int cluster, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * cluster));
  cfg.blockDim = dim3(kResolveThreads);
  cfg.dynamicSmemBytes = resolve_smem(p);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, chain_resolve_kernel<BF16>, p);
}

// A kernel of `threads`-thread CTAs launched as a programmatic dependent of
// the kernel before it.
template <typename Kern, typename... Args>
cudaError_t launch_dependent(Kern k, dim3 grid, int threads, size_t smem, cudaStream_t s,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

cudaError_t launch_generation(const ChainStochParams &p, cudaStream_t s) {
  return launch_dependent(advance_generation_kernel, dim3(1), 1, 0, s, p.gen, p.claim);
}

// The plain verify: the generation step, the bulk-copy ring stream, then the
// resolve kernel, each a programmatic dependent of the one before.
template <bool BF16, int S>
cudaError_t launch_t(const ChainStochParams &p, int grid, size_t smem, int cluster, cudaStream_t s) {
  cudaError_t e = prepare<BF16>(cluster);
  if (e == cudaSuccess) e = prepare_ring<BF16, kSoftVecs, S>(smem);
  if (e != cudaSuccess) return e;
  e = launch_generation(p, s);
  if (e == cudaSuccess)
    e = launch_dependent(softmax_partials_kernel<BF16, kSoftVecs, S, false>, dim3(static_cast<unsigned>(grid)),
                         kSoftThreads + 32, smem, s, p);
  if (e == cudaSuccess) e = launch_resolve<BF16>(p, cluster, s);
  return e;
}

template <bool BF16, int S>
cudaError_t ring_blocks_t(size_t smem, int *blocks) {
  cudaError_t e = prepare_ring<BF16, kSoftVecs, S>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, softmax_partials_kernel<BF16, kSoftVecs, S, false>,
                                                       kSoftThreads + 32, smem);
}

// The truncated verify: the generation step, the ring stream with its chunk
// maxima (always kSoftStages deep), the selection kernel, then the resolve
// kernel, each a programmatic dependent of the one before.
template <bool BF16>
cudaError_t launch_truncated_t(const ChainStochParams &p, int grid, size_t smem, int cluster,
                               cudaStream_t s) {
  cudaError_t e = prepare<BF16>(cluster);
  if (e == cudaSuccess) e = prepare_ring<BF16, kSoftVecs, kSoftStages, true>(smem);
  if (e != cudaSuccess) return e;
  const dim3 rows(static_cast<unsigned>(p.B * (2 * p.K + 1)));
  e = launch_generation(p, s);
  if (e == cudaSuccess)
    e = launch_dependent(softmax_partials_kernel<BF16, kSoftVecs, kSoftStages, true>,
                         dim3(static_cast<unsigned>(grid)), kSoftThreads + 32, smem, s, p);
  if (e == cudaSuccess) e = launch_dependent(trunc_select_kernel<BF16>, rows, kSelThreads, 0, s, p);
  if (e == cudaSuccess) e = launch_resolve<BF16>(p, cluster, s);
  return e;
}

// DRIFT: the generation step, the ring stream over positions 0 .. K-1 (with
// the target rows' chunk maxima), one pick CTA per drafted position (the
// top m of its target row), then one CTA per row that forms the residuals
// and the row status, each a programmatic dependent of the one before.
template <bool BF16>
cudaError_t launch_drift_t(const ChainStochParams &p, int grid, size_t smem, cudaStream_t s) {
  cudaError_t e = prepare_ring<BF16, kSoftVecs, kSoftStages, true>(smem);
  if (e != cudaSuccess) return e;
  e = launch_generation(p, s);
  if (e == cudaSuccess)
    e = launch_dependent(softmax_partials_kernel<BF16, kSoftVecs, kSoftStages, true>,
                         dim3(static_cast<unsigned>(grid)), kSoftThreads + 32, smem, s, p);
  if (e == cudaSuccess)
    e = launch_dependent(drift_pick_kernel<BF16>, dim3(static_cast<unsigned>(p.B * p.K)), kSelThreads, 0, s, p);
  if (e == cudaSuccess)
    e = launch_dependent(drift_finish_kernel<BF16>, dim3(static_cast<unsigned>(p.B)), kDriftFinishThreads, 0, s, p);
  return e;
}

}  // namespace

#ifdef SV_BOUNDS
SV_OOB_READER(oob_record_chain)

// The checker's own check: one thread tests index 5 against an extent of 3
// (nothing is read or written there), which must leave one record.
__global__ void oob_selftest_kernel() { (void)SV_INB(5, 3); }

cudaError_t oob_selftest(cudaStream_t s) {
  oob_selftest_kernel<<<1, 1, 0, s>>>();
  return cudaGetLastError();
}
#endif

cudaError_t launch_chain_stochastic(const ChainStochParams &p, bool bf16, int grid, size_t smem,
                                    int cluster, cudaStream_t s) {
  if (p.stages == 4)
    return bf16 ? launch_t<true, 4>(p, grid, smem, cluster, s) : launch_t<false, 4>(p, grid, smem, cluster, s);
  if (p.stages == 3)
    return bf16 ? launch_t<true, 3>(p, grid, smem, cluster, s) : launch_t<false, 3>(p, grid, smem, cluster, s);
  return bf16 ? launch_t<true, 2>(p, grid, smem, cluster, s) : launch_t<false, 2>(p, grid, smem, cluster, s);
}

cudaError_t ring_blocks_per_sm(bool bf16, int stages, size_t smem, int *blocks) {
  if (stages == 4) return bf16 ? ring_blocks_t<true, 4>(smem, blocks) : ring_blocks_t<false, 4>(smem, blocks);
  if (stages == 3) return bf16 ? ring_blocks_t<true, 3>(smem, blocks) : ring_blocks_t<false, 3>(smem, blocks);
  return bf16 ? ring_blocks_t<true, 2>(smem, blocks) : ring_blocks_t<false, 2>(smem, blocks);
}

cudaError_t launch_chain_truncated(const ChainStochParams &p, bool bf16, int grid, size_t smem,
                                   int cluster, cudaStream_t s) {
  return bf16 ? launch_truncated_t<true>(p, grid, smem, cluster, s)
              : launch_truncated_t<false>(p, grid, smem, cluster, s);
}

cudaError_t launch_drift(const ChainStochParams &p, bool bf16, int grid, size_t smem, cudaStream_t s) {
  return bf16 ? launch_drift_t<true>(p, grid, smem, s) : launch_drift_t<false>(p, grid, smem, s);
}

}  // namespace sv
