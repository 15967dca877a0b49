// chain_stochastic.cu -- the stochastic chain verifier (one kernel per step).
//
// Computes, for every row b and draft position j, the tests of
// "Speculative Decoding: Draft, Verify, and Correct" ('Name the two
// distributions at one prefix', 'Verify several proposed tokens in one target
// pass'): p = softmax(target/T), q = softmax(draft/T), accept y_j iff
// p(y_j)/q(y_j) >= 1 or u < p(y_j)/q(y_j); at a rejection draw from
// [p - q]+ by inverse CDF; at j = K draw the bonus from p.  The walk to the
// first rejection is fused in as a "last position of the row finishes" step.
//
// Layout of the work: a persistent grid of thread-block clusters of C CTAs.
// Each cluster owns a round-robin share of the B*(K+1) positions; CTA r of the
// cluster owns vocabulary slice [r*L, (r+1)*L) of each position.  Per position:
//   1. bulk copies (TMA, non-multicast) of the CTA's target and draft slices
//      land in a `stages`-deep shared-memory ring, prefetched ahead;
//   2. pass 1 moves the slice to registers and finds the NaN-propagating max;
//      max exchanged across the cluster through distributed shared memory;
//   3. pass 2 turns every logit into exp2((x - max) * log2(e) / T) in place
//      (one exp per logit, kept in registers) and sums; sums exchanged;
//   4. the acceptance ratio is formed in log2 space from the draft token's
//      logits; a rejecting position sums its residual [p - q]+ from the
//      registers (no more exps, no more HBM traffic), exchanges the per-CTA
//      masses, and the CTA whose range holds u * Z finds the token with a
//      hierarchical scan (round -> warp -> lane -> element, vocabulary order).
// Every logit is read from HBM exactly once.
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace sv {
namespace {

constexpr int NT = kThreads;
constexpr int NW = NT / 32;
constexpr int kMaxNV = 8;
constexpr int kMaxStages = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInf = __builtin_huge_valf();

struct alignas(16) Ctrl {
  uint64_t full[kMaxStages];  // stage "data landed" barriers
  uint64_t never;             // a barrier nothing completes (forced-timeout test)
  uint64_t pad0;
  float4 mailbox[2];          // this CTA's slot of the cluster exchange (double buffered)
  float4 part[NW];            // block-reduction partials
  float wtot[kMaxNV][NW];     // inverse-CDF search: per-round warp totals
  float sel_t;                // search: remainder handed to the chosen warp
  int sel[3];                 // search: chosen round, warp, element
};
static_assert(sizeof(Ctrl) <= 2048, "control block must fit its reservation");

template <bool BF16>
struct Fmt {
  static constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr uint32_t NEG_INF_WORD = BF16 ? 0xFF80FF80u : 0xFF800000u;
  // element e of a 16-byte vector held as 4 words
  static __device__ __forceinline__ float elem(const uint32_t *w, int e) {
    if constexpr (BF16) return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
    else return __uint_as_float(w[e]);
  }
  // set elements [valid, EPV) to -inf
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
  static __device__ __forceinline__ float load_logit(const void *base, size_t idx) {
    if constexpr (BF16)
      return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short *>(base) + idx)) << 16);
    else return __ldg(static_cast<const float *>(base) + idx);
  }
  // One vector of the slice: from the shared-memory stage (bulk-copy path) or
  // straight from global memory (unaligned rows).  Elements >= len are -inf.
  static __device__ __forceinline__ void load_vec(uint32_t *w, bool tma, const unsigned char *sbuf,
                                                  const char *gsrc, int v, int len) {
    const int valid = len - v * EPV;
    if (valid <= 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = NEG_INF_WORD;
      return;
    }
    if (tma) {
      uint4 r = ld_shared_u4(sbuf + (size_t)v * 16);
      w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
          const int e0 = v * 8 + 2 * i;
          const unsigned short *g = reinterpret_cast<const unsigned short *>(gsrc);
          uint32_t lo = e0 < len ? __ldg(g + e0) : 0xFF80u;
          uint32_t hi = e0 + 1 < len ? __ldg(g + e0 + 1) : 0xFF80u;
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

// Block reduction of two floats; result valid in thread 0.  `op` combines.
template <class Op>
__device__ __forceinline__ float2 block_reduce2(float a, float b, float ident, Op op, Ctrl &ctl,
                                                int lane, int warp) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = op(a, __shfl_xor_sync(FULL_MASK, a, o));
    b = op(b, __shfl_xor_sync(FULL_MASK, b, o));
  }
  if (lane == 0) ctl.part[warp] = make_float4(a, b, 0.f, 0.f);
  __syncthreads();
  float2 r = make_float2(ident, ident);
  if (warp == 0) {
    if (lane < NW) {
      float4 v = ctl.part[lane];
      r = make_float2(v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      r.x = op(r.x, __shfl_xor_sync(FULL_MASK, r.x, o));
      r.y = op(r.y, __shfl_xor_sync(FULL_MASK, r.y, o));
    }
  }
  return r;
}

// Publish this CTA's value in mailbox[slot], then every warp fetches the C
// values of the cluster: lane c (< C) holds CTA c's value on return.
__device__ __forceinline__ float4 cluster_exchange(float4 mine, Ctrl &ctl, int slot, uint32_t C,
                                                   int tid, int lane) {
  if (tid == 0) ctl.mailbox[slot] = mine;
  cluster_sync();
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane < (int)C) v = ld_dsmem_f4(dsmem_addr(&ctl.mailbox[slot], (uint32_t)lane));
  return v;
}

// Choose the CTA whose cumulative interval (CTA order = vocabulary order)
// holds u * total of the per-CTA masses held by lanes 0..C-1.  Returns the CTA
// (or -1 without mass) and the remainder inside it (+inf: clamp to the last
// positive entry of that CTA).
__device__ __forceinline__ int cluster_pick(float mass_lane, uint32_t C, float u, float *t_local,
                                            float *total) {
  float Z = 0.f;
  for (uint32_t c = 0; c < C; ++c) Z += __shfl_sync(FULL_MASK, mass_lane, c);
  const float t = u * Z;
  float acc = 0.f, tl = 0.f;
  int cs = -1, clast = -1;
  for (uint32_t c = 0; c < C; ++c) {
    const float m = __shfl_sync(FULL_MASK, mass_lane, c);
    const float prev = acc;
    acc += m;
    if (m > 0.f) clast = (int)c;
    if (cs < 0 && m > 0.f && acc > t) {
      cs = (int)c;
      tl = t - prev;
    }
  }
  if (cs < 0) {
    cs = clast;
    tl = kInf;
  }
  *t_local = tl;
  *total = Z;
  return cs;
}

// Inverse CDF inside one CTA: the slice-local index of the element whose
// cumulative interval (vocabulary order) holds t, masses mass(i) for register
// slot i = k*EPV + e (element (tid + k*NT)*EPV + e of the slice).  t = +inf
// or a t past the total picks the last element with positive mass.  Every
// level (round, warp, lane, element) uses intervals built from the same sums
// it compares against, so the choice always lands on positive mass.
template <int NV, int EPV, class F>
__device__ __forceinline__ int cta_inverse_cdf(float t, F mass, Ctrl &ctl, int tid, int lane,
                                               int warp) {
  float rs[NV], incl[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    float r = 0.f;
#pragma unroll
    for (int e = 0; e < EPV; ++e) r += mass(k * EPV + e);
    rs[k] = r;
    incl[k] = warp_inclusive_scan(r, lane);
    if (lane == 31) ctl.wtot[k][warp] = incl[k];
  }
  __syncthreads();
  if (tid == 0) {
    float acc = 0.f, t2 = 0.f;
    int ks = -1, ws = -1;
    for (int k = 0; k < NV && ks < 0; ++k)
      for (int w = 0; w < NW; ++w) {
        const float m = ctl.wtot[k][w];
        const float prev = acc;
        acc += m;
        if (m > 0.f && acc > t) {
          ks = k;
          ws = w;
          t2 = t - prev;
          break;
        }
      }
    if (ks < 0) {
      for (int k = NV - 1; k >= 0 && ks < 0; --k)
        for (int w = NW - 1; w >= 0; --w)
          if (ctl.wtot[k][w] > 0.f) {
            ks = k;
            ws = w;
            t2 = kInf;
            break;
          }
    }
    ctl.sel[0] = ks;
    ctl.sel[1] = ws;
    ctl.sel[2] = -1;
    ctl.sel_t = t2;
  }
  __syncthreads();
  const int ks = ctl.sel[0], ws = ctl.sel[1];
  const float t2 = ctl.sel_t;
  if (ks >= 0 && warp == ws) {
    float my_incl = 0.f, my_r = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (k == ks) {
        my_incl = incl[k];
        my_r = rs[k];
      }
    float excl = __shfl_up_sync(FULL_MASK, my_incl, 1);
    if (lane == 0) excl = 0.f;
    const unsigned hit = __ballot_sync(FULL_MASK, my_r > 0.f && my_incl > t2);
    int ls;
    bool clamp = false;
    if (hit) {
      ls = __ffs(hit) - 1;
    } else {
      const unsigned pos = __ballot_sync(FULL_MASK, my_r > 0.f);
      ls = 31 - __clz(pos);
      clamp = true;
    }
    if (lane == ls) {
      const float t3 = clamp ? kInf : t2 - excl;
      float c = 0.f;
      int es = -1, elast = -1;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (k == ks) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float m = mass(k * EPV + e);
            c += m;
            if (m > 0.f) {
              elast = e;
              if (es < 0 && c > t3) es = e;
            }
          }
        }
      if (es < 0) es = elast;
      ctl.sel[2] = (tid + ks * NT) * EPV + es;
    }
  }
  __syncthreads();
  return ctl.sel[2];
}

// Row walk of "Verify several proposed tokens in one target pass": first
// rejecting position, then the emitted tokens.  One warp.
__device__ void walk_chain_row(const ChainStochParams &P, int b, int lane) {
  const int K = P.K, npos = K + 1;
  const ChainRec *R = P.rec + (size_t)b * npos;
  uint32_t flags = 0;
  int stop = K;
  for (int j0 = 0; j0 < npos; j0 += 32) {
    const int j = j0 + lane;
    int acc = 1;
    if (j < npos) {
      const int4 r = __ldcg(reinterpret_cast<const int4 *>(R + j));
      flags |= static_cast<uint32_t>(r.z);
      if (j < K) acc = r.y;
    }
    const unsigned rej = __ballot_sync(FULL_MASK, !acc);
    if (stop == K && rej) stop = j0 + __ffs(rej) - 1;
  }
  flags = __reduce_or_sync(FULL_MASK, flags);
  const int tok = __ldcg(&R[stop].token);
  for (int j = lane; j < npos; j += 32) {
    int o = -1;
    if (!flags) o = j < stop ? __ldg(P.tokens + (size_t)b * K + j) : (j == stop ? tok : -1);
    P.out_tokens[(size_t)b * npos + j] = o;
  }
  if (lane == 0) {
    P.accepted_len[b] = flags ? -1 : stop;
    P.num_emitted[b] = flags ? 0 : stop + 1;
    P.row_status[b] = lowest_code(flags);
    P.row_counter[b] = 0u;  // leave the workspace zero-filled for the next call
  }
}

template <bool BF16, int NV>
__global__ void __launch_bounds__(NT, 1) chain_stochastic_kernel(const __grid_constant__ ChainStochParams P) {
  using F = Fmt<BF16>;
  constexpr int EPV = F::EPV;
  constexpr int E = NV * EPV;
  constexpr int ESZ = F::ESZ;
  static_assert(E <= kMaxElemsPerThread, "register budget");

  extern __shared__ __align__(128) unsigned char smem[];
  const int S = P.stages;
  Ctrl &ctl = *reinterpret_cast<Ctrl *>(smem + (size_t)S * 2 * P.buf_bytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_ctarank(), C = cluster_nctarank();
  const int cid = (int)cluster_id_x(), NC = (int)num_clusters_x();
  const int B = P.B, K = P.K, V = P.V, npos = K + 1;
  const int W = B * npos;
  const int my_items = cid < W ? (W - 1 - cid) / NC + 1 : 0;
  const int s0 = (int)crank * P.L;
  const int len = max(0, min(V, s0 + P.L) - s0);
  const bool tma = P.use_tma != 0;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&ctl.full[s], 1);
    mbar_init(&ctl.never, 1);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // every CTA of the cluster is running: DSMEM may be used from here on

  auto decode = [&](int n, int &b, int &j) {  // drafts first (heavier), bonus rows last
    const int it = cid + n * NC;
    if (it < B * K) {
      b = it / K;
      j = it - b * K;
    } else {
      b = it - B * K;
      j = K;
    }
  };
  const uint64_t pol = l2_policy_evict_first();
  auto issue = [&](int n) {  // thread 0: bulk copies of item n into stage n % S
    int b, j;
    decode(n, b, j);
    const int s = n % S;
    unsigned char *tb = smem + (size_t)s * 2 * P.buf_bytes;
    const uint32_t bytes = static_cast<uint32_t>(len) * ESZ;
    mbar_arrive_expect_tx(&ctl.full[s], bytes * (j < K ? 2u : 1u));
    if (bytes) {
      bulk_g2s(tb, static_cast<const char *>(P.target) + ((size_t)(b * npos + j) * V + s0) * ESZ,
               bytes, &ctl.full[s], pol);
      if (j < K)
        bulk_g2s(tb + P.buf_bytes,
                 static_cast<const char *>(P.draft) + ((size_t)(b * K + j) * V + s0) * ESZ, bytes,
                 &ctl.full[s], pol);
    }
  };

  int issued = 0;     // thread 0: items whose copies were issued
  int n_break = -1;   // first item whose wait gave up (CTA-uniform)
  if (tma && tid == 0)
    for (; issued < min(S, my_items); ++issued) issue(issued);

  int xslot = 0;
  for (int n = 0; n < my_items; ++n) {
    int b, j;
    decode(n, b, j);
    const int s = n % S;
    const uint32_t parity = static_cast<uint32_t>(n / S) & 1u;

    // ---- item scalars (identical in every CTA of the cluster)
    uint32_t iflags = 0;
    const float T = P.temperature ? __ldg(P.temperature + b) : 1.0f;
    if (!(T > 0.f && T < kInf)) iflags |= F_BAD_TEMPERATURE;
    const float s2 = (iflags & F_BAD_TEMPERATURE) ? 1.f : __fdiv_rn(kLog2e, T);
    const float u_s = __ldg(P.u_sample + (size_t)b * npos + j);
    if (!(u_s >= 0.f && u_s < 1.f)) iflags |= F_BAD_UNIFORM;
    int y = 0;
    float u_a = 0.f, a_y = 0.f, b_y = 0.f;
    if (j < K) {
      y = __ldg(P.tokens + (size_t)b * K + j);
      u_a = __ldg(P.u_accept + (size_t)b * K + j);
      if (!(u_a >= 0.f && u_a < 1.f)) iflags |= F_BAD_UNIFORM;
      if (y < 0 || y >= V) {
        iflags |= F_BAD_TOKEN;
        y = 0;
      }
      a_y = F::load_logit(P.target, (size_t)(b * npos + j) * V + y);
      b_y = F::load_logit(P.draft, (size_t)(b * K + j) * V + y);
    }

    // ---- wait for the slices (bounded)
    bool timed_out = false;
    if (tma && n_break < 0)
      timed_out = P.force_timeout ? !mbar_wait_bounded(&ctl.never, 0u, P.wait_limit_ns)
                                  : !mbar_wait_bounded(&ctl.full[s], parity, P.wait_limit_ns);

    // ---- pass 1: slice -> registers, NaN-propagating max
    const unsigned char *tb = smem + (size_t)s * 2 * P.buf_bytes;
    const char *tg = static_cast<const char *>(P.target) + ((size_t)(b * npos + j) * V + s0) * ESZ;
    const char *dg = static_cast<const char *>(P.draft) + ((size_t)(b * K + j) * V + s0) * ESZ;
    uint32_t wp[NV * 4], wq[NV * 4];
    float mp = -kInf, mq = -kInf;
    {
      uint32_t pmp = F::NEG_INF_WORD, pmq = F::NEG_INF_WORD;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        F::load_vec(wp + 4 * k, tma, tb, tg, tid + k * NT, len);
        if constexpr (BF16) {
#pragma unroll
          for (int i = 0; i < 4; ++i) pmp = bf16x2_max_nan(pmp, wp[4 * k + i]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) mp = fmax_nan(mp, __uint_as_float(wp[4 * k + i]));
        }
      }
      if (j < K) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          F::load_vec(wq + 4 * k, tma, tb + P.buf_bytes, dg, tid + k * NT, len);
          if constexpr (BF16) {
#pragma unroll
            for (int i = 0; i < 4; ++i) pmq = bf16x2_max_nan(pmq, wq[4 * k + i]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) mq = fmax_nan(mq, __uint_as_float(wq[4 * k + i]));
          }
        }
      }
      if constexpr (BF16) {
        mp = fmax_nan(bf16_lo(pmp), bf16_hi(pmp));
        mq = fmax_nan(bf16_lo(pmq), bf16_hi(pmq));
      }
    }
    // everyone has read stage s; a wait that gave up anywhere breaks the pipeline
    if (__syncthreads_or(timed_out) && n_break < 0) n_break = n;
    if (n_break >= 0) iflags |= F_TIMEOUT;
    if (tma && tid == 0 && n_break < 0 && issued < my_items) issue(issued++);

    // ---- exchange 1: max of p and q logits, row flags
    float4 xv;
    {
      const float2 r = block_reduce2(mp, mq, -kInf, fmax_nan, ctl, lane, warp);
      xv = cluster_exchange(make_float4(r.x, r.y, __uint_as_float(iflags), 0.f), ctl, xslot, C,
                            tid, lane);
      xslot ^= 1;
    }
    float Mp = -kInf, Mq = -kInf;
    uint32_t flags = 0;
    for (uint32_t c = 0; c < C; ++c) {
      Mp = fmax_nan(Mp, __shfl_sync(FULL_MASK, xv.x, c));
      Mq = fmax_nan(Mq, __shfl_sync(FULL_MASK, xv.y, c));
      flags |= __float_as_uint(__shfl_sync(FULL_MASK, xv.z, c));
    }
    if (Mp != Mp || Mp == kInf) flags |= F_NONFINITE;
    else if (Mp == -kInf) flags |= F_EMPTY;
    if (j < K) {
      if (Mq != Mq || Mq == kInf) flags |= F_NONFINITE;
      else if (Mq == -kInf) flags |= F_EMPTY;
    }

    int owner = 0, token = -1, accept = (j < K) ? 0 : 1;
    float p_y = 0.f, q_y = 0.f, Z = 0.f;
    if (!flags) {
      // ---- pass 2: exp2 in registers, sums
      const float nMp = -__fmul_rn(Mp, s2), nMq = -__fmul_rn(Mq, s2);
      float ep[E], eq[E];
      float sp = 0.f, sq = 0.f;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        float r = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          ep[k * EPV + e] = ex2(__fmaf_rn(F::elem(wp + 4 * k, e), s2, nMp));
          r += ep[k * EPV + e];
        }
        sp += r;
      }
      if (j < K) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          float r = 0.f;
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            eq[k * EPV + e] = ex2(__fmaf_rn(F::elem(wq + 4 * k, e), s2, nMq));
            r += eq[k * EPV + e];
          }
          sq += r;
        }
      }
      // ---- exchange 2: partition sums
      const float2 r2 = block_reduce2(sp, sq, 0.f, [](float a, float c) { return a + c; }, ctl,
                                      lane, warp);
      const float4 sv = cluster_exchange(make_float4(r2.x, r2.y, 0.f, 0.f), ctl, xslot, C, tid,
                                         lane);
      xslot ^= 1;
      float Sp = 0.f, Sq = 0.f;
      for (uint32_t c = 0; c < C; ++c) {
        Sp += __shfl_sync(FULL_MASK, sv.x, c);
        Sq += __shfl_sync(FULL_MASK, sv.y, c);
      }

      int search = 0;  // 0: none, 1: residual [p - q]+, 2: target law p
      float mass_lane = sv.x;
      if (j < K) {
        // ratio p(y)/q(y) in log2 space: identical logits give exactly 0
        const float l2p = __fadd_rn(__fmaf_rn(a_y, s2, nMp), -lg2(Sp));
        const float l2q = __fadd_rn(__fmaf_rn(b_y, s2, nMq), -lg2(Sq));
        const float l2r = __fadd_rn(l2p, -l2q);
        accept = (l2r >= 0.f) || (u_a < ex2(l2r));
        p_y = ex2(l2p);
        q_y = ex2(l2q);
        if (!accept) {
          const float iSp = __frcp_rn(Sp), iSq = __frcp_rn(Sq);
          float rsum = 0.f;
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            float r = 0.f;
#pragma unroll
            for (int e = 0; e < EPV; ++e)
              r += fmaxf(__fmaf_rn(ep[k * EPV + e], iSp, -__fmul_rn(eq[k * EPV + e], iSq)), 0.f);
            rsum += r;
          }
          // ---- exchange 3: residual mass per CTA
          const float2 r3 = block_reduce2(rsum, 0.f, 0.f, [](float a, float c) { return a + c; },
                                          ctl, lane, warp);
          const float4 rv = cluster_exchange(make_float4(r3.x, 0.f, 0.f, 0.f), ctl, xslot, C, tid,
                                             lane);
          xslot ^= 1;
          float tl_unused, Zr;
          cluster_pick(rv.x, C, 0.f, &tl_unused, &Zr);
          Z = Zr;
          if (Z > 0.f) {
            search = 1;
            mass_lane = rv.x;
          } else {
            search = 2;  // residual vanished in fp32: draw from p
          }
          if (search == 1) {
            float tl, tot;
            owner = cluster_pick(mass_lane, C, u_s, &tl, &tot);
            if ((int)crank == owner) {
              const int li = cta_inverse_cdf<NV, EPV>(
                  tl,
                  [&](int i) {
                    return fmaxf(__fmaf_rn(ep[i], iSp, -__fmul_rn(eq[i], iSq)), 0.f);
                  },
                  ctl, tid, lane, warp);
              token = s0 + li;
            }
          }
        }
      } else {
        search = 2;  // bonus
      }
      if (search == 2) {
        float tl, tot;
        owner = cluster_pick(sv.x, C, u_s, &tl, &tot);
        if ((int)crank == owner) {
          const int li = cta_inverse_cdf<NV, EPV>(tl, [&](int i) { return ep[i]; }, ctl, tid, lane,
                                                  warp);
          token = s0 + li;
        }
      }
    }

    // ---- record, diagnostics, and the row walk by the last position to finish
    if (owner < 0) owner = 0;  // never leave a position without a writer
    if ((int)crank == owner && warp == 0) {
      unsigned old = 0;
      if (lane == 0) {
        const size_t o = (size_t)b * npos + j;
        __stcg(reinterpret_cast<int4 *>(P.rec + o),
               make_int4(token, accept, static_cast<int>(flags), 0));
        if (j < K) {
          const size_t d = (size_t)b * K + j;
          if (P.p_at_draft) P.p_at_draft[d] = p_y;
          if (P.q_at_draft) P.q_at_draft[d] = q_y;
          if (P.resid_mass) P.resid_mass[d] = accept ? 0.f : Z;
        }
        __threadfence();
        old = atomicAdd(P.row_counter + b, 1u);
      }
      old = __shfl_sync(FULL_MASK, old, 0);
      if (old == static_cast<unsigned>(K)) {
        __threadfence();
        walk_chain_row(P, b, lane);
      }
    }
  }

  // copies issued after a wait gave up may still be landing: let them finish
  if (tma && n_break >= 0 && tid == 0)
    for (int m = n_break; m < issued; ++m)
      mbar_wait_bounded(&ctl.full[m % S], static_cast<uint32_t>(m / S) & 1u, P.wait_limit_ns);
  __syncthreads();
  cluster_sync();  // no CTA leaves while a peer may still read its mailbox
}

// Function attributes are set once per device (and again only when a larger
// shared-memory size is needed), so steady-state launches make no driver
// calls besides the launch itself and can be captured into a CUDA graph.
template <bool BF16, int NV>
cudaError_t prepare(size_t smem, int cluster) {
  static std::atomic<size_t> done_smem[kMaxDevices];
  static std::atomic<int> done_nonportable[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  auto k = chain_stochastic_kernel<BF16, NV>;
  if (done_smem[dev].load() < smem) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    done_smem[dev].store(smem);
  }
  if (cluster > 8 && !done_nonportable[dev].load()) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    done_nonportable[dev].store(1);
  }
  return cudaSuccess;
}

template <bool BF16, int NV>
cudaError_t launch_t(const ChainStochParams &p, int cluster, int grid_clusters, size_t smem,
                     cudaStream_t s) {
  cudaError_t e = prepare<BF16, NV>(smem, cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster * grid_clusters));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, chain_stochastic_kernel<BF16, NV>, p);
}

template <bool BF16, int NV>
cudaError_t max_clusters_t(int cluster, size_t smem, int *out) {
  cudaError_t e = prepare<BF16, NV>(smem, cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster * 64));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, chain_stochastic_kernel<BF16, NV>, &cfg);
}

}  // namespace

cudaError_t launch_chain_stochastic(const ChainStochParams &p, bool bf16, int nv, int cluster,
                                    int grid_clusters, size_t smem, cudaStream_t s) {
  if (bf16) {
    switch (nv) {
      case 1: return launch_t<true, 1>(p, cluster, grid_clusters, smem, s);
      case 2: return launch_t<true, 2>(p, cluster, grid_clusters, smem, s);
      case 4: return launch_t<true, 4>(p, cluster, grid_clusters, smem, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (nv) {
    case 1: return launch_t<false, 1>(p, cluster, grid_clusters, smem, s);
    case 2: return launch_t<false, 2>(p, cluster, grid_clusters, smem, s);
    case 4: return launch_t<false, 4>(p, cluster, grid_clusters, smem, s);
    case 8: return launch_t<false, 8>(p, cluster, grid_clusters, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t chain_stochastic_max_clusters(bool bf16, int nv, int cluster, size_t smem,
                                          int *clusters) {
  if (bf16) {
    switch (nv) {
      case 1: return max_clusters_t<true, 1>(cluster, smem, clusters);
      case 2: return max_clusters_t<true, 2>(cluster, smem, clusters);
      case 4: return max_clusters_t<true, 4>(cluster, smem, clusters);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (nv) {
    case 1: return max_clusters_t<false, 1>(cluster, smem, clusters);
    case 2: return max_clusters_t<false, 2>(cluster, smem, clusters);
    case 4: return max_clusters_t<false, 4>(cluster, smem, clusters);
    case 8: return max_clusters_t<false, 8>(cluster, smem, clusters);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sv
