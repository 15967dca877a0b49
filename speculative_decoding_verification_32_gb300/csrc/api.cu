// api.cu -- the C ABI of include/specverify.h: argument validation (before
// any CUDA call), launch-shape selection from the device's occupancy, and the
// launches.  No allocation, no synchronisation.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "internal.h"
#include "specverify.h"

using namespace sv;

// Scratch of spec_verify_chain_static: part of the library image, one copy
// per device, so that entry point never allocates.
static __device__ __align__(256) unsigned char g_static_ws[SPEC_STATIC_WS_BYTES];

namespace {

std::atomic<uint64_t> g_wait_ns{1000000000ull};
std::atomic<int> g_force_timeout{0};

struct DevInfo {
  int sms = 0;
  int smem_optin = 0;
  int l2_bytes = 0;
};

std::mutex g_mu;
std::map<int, DevInfo> g_dev;
std::map<std::tuple<int, int, size_t>, int> g_blocks;
std::map<std::tuple<int, int, int>, int> g_greedy_blocks;
void *g_static_ws_ptr[kMaxDevices] = {};  // device address of g_static_ws, per device

constexpr int kMinGreedySlice = 2048;
constexpr size_t kRingCtrlBytes = 2048;  // the ring stream kernel's control block

// SPECVERIFY_VERBOSE=1 prints each distinct launch shape once (stderr).
void report(const char *what, long long a, long long b, long long c, long long d, long long e,
            long long f, long long g) {
  static const bool on = [] {
    const char *v = std::getenv("SPECVERIFY_VERBOSE");
    return v && *v && *v != '0';
  }();
  if (!on) return;
  static std::mutex mu;
  static std::map<std::tuple<std::string, long long, long long, long long, long long, long long,
                             long long, long long>, int> seen;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_tuple(std::string(what), a, b, c, d, e, f, g);
  if (seen.count(key)) return;
  seen[key] = 1;
  std::fprintf(stderr, "[specverify] %s: %lld %lld %lld %lld %lld %lld %lld\n", what, a, b, c, d,
               e, f, g);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned(const void *p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }
int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

cudaError_t device_info(int *dev, DevInfo *info) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_dev.find(*dev);
  if (it != g_dev.end()) {
    *info = it->second;
    return cudaSuccess;
  }
  DevInfo d;
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, *dev);
  if (e != cudaSuccess) return e;
  g_dev[*dev] = d;
  *info = d;
  return cudaSuccess;
}

cudaError_t ring_blocks(int dev, bool bf16, int stages, size_t smem, int *out) {
  auto key = std::make_tuple(dev, 8 + (int)bf16 + 2 * stages, smem);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_blocks.find(key);
    if (it != g_blocks.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  cudaError_t e = ring_blocks_per_sm(bf16, stages, smem, out);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  g_blocks[key] = *out;
  return cudaSuccess;
}

cudaError_t greedy_blocks(int dev, bool bf16, bool vec, int *out) {
  auto key = std::make_tuple(dev, (int)bf16, (int)vec);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_greedy_blocks.find(key);
    if (it != g_greedy_blocks.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  cudaError_t e = greedy_max_blocks_per_sm(bf16, vec, out);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  g_greedy_blocks[key] = *out;
  return cudaSuccess;
}

size_t greedy_partials_max(int32_t B, int32_t npos, int32_t V) {
  return static_cast<size_t>(B) * npos * ceil_div(V, kMinGreedySlice) * sizeof(GreedyPart);
}

// The truncated verify's chunk maxima, after the records: 2 bytes per
// (logit row, ring tile, consumer thread), for the fp32 tiling (the one with
// more tiles).
size_t chunk_max_bytes(size_t rows, int32_t V) {
  return align_up(rows * ceil_div(V, kSoftMinSlice) * kSoftThreads * 2, 256);
}

bool valid_sizes(int32_t B, int32_t V) { return B >= 0 && V >= 1 && V <= SPEC_MAX_V; }

// Greedy launch shared by the chain (GREEDY mode) and tree entry points.
// The slice (elements per work item) is picked from 2048..16384 to minimise
// the busiest warp's load: rounds of items per warp times (slice bytes + a
// fixed per-item cost of about 2 KB of streaming).
spec_status run_greedy(GreedyParams &p, bool bf16, int esz, void *ws, cudaStream_t stream) {
  int dev;
  DevInfo di;
  if (device_info(&dev, &di) != cudaSuccess) return SPEC_ERR_CUDA;
  p.vec = aligned(p.target, 16) && (static_cast<long long>(p.V) * esz) % 16 == 0;
  int per_sm = 0;
  if (greedy_blocks(dev, bf16, p.vec != 0, &per_sm) != cudaSuccess || per_sm < 1) return SPEC_ERR_CUDA;
  const long long warps = static_cast<long long>(di.sms) * per_sm * (kGreedyThreads / 32);
  const long long positions = static_cast<long long>(p.B) * p.npos;
  int slice = kGreedySlice;
  double best_cost = 0.0;
  for (int sl = kGreedySlice; sl >= kMinGreedySlice; sl /= 2) {
    const long long items = positions * ceil_div(p.V, sl);
    const double cost = static_cast<double>((items + warps - 1) / warps) *
                        (static_cast<double>(std::min(sl, p.V)) * esz + 2048.0);
    if (sl == kGreedySlice || cost < best_cost) {
      best_cost = cost;
      slice = sl;
    }
  }
  // SPECVERIFY_GREEDY_SLICE (2048..16384 elements) overrides it for tuning
  if (const char *ov = std::getenv("SPECVERIFY_GREEDY_SLICE")) {
    const int sl = std::atoi(ov);
    if (sl >= kMinGreedySlice && sl <= kGreedySlice) slice = static_cast<int>(align_up(static_cast<size_t>(sl), 8));
  }
  p.slice = slice;
  p.nslices = ceil_div(p.V, slice);
  p.part = static_cast<GreedyPart *>(ws);
  const long long items = positions * p.nslices;
  if (items > 0x7fffffffLL) return SPEC_ERR_SHAPE;
  const long long need = (items + kGreedyThreads / 32 - 1) / (kGreedyThreads / 32);
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(need, static_cast<long long>(di.sms) * per_sm)));
  report("greedy slice nslices per_sm grid vec", slice, p.nslices, per_sm, grid, p.vec, 0, 0);
  if (launch_greedy(p, bf16, grid, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

// The stochastic calls' stream is the bulk-copy ring: the plain verify's, or
// the one that also keeps chunk maxima (truncated verify and DRIFT), which is
// always kSoftStages deep.
enum class StreamKind { kRing, kRingListed };

// Parameters and launch shapes of the stochastic stream kernel and of the
// resolve kernel's cluster split, from the arguments and the workspace;
// output pointers are left for the caller.
spec_status setup_stochastic(const spec_chain_args *a, void *ws, size_t ws_bytes, ChainStochParams &p,
                             int &grid, int &C, StreamKind kind, size_t *smem) {
  const int K = a->K;
  const int esz = a->dtype == SPEC_BF16 ? 2 : 4;
  const bool bf16 = a->dtype == SPEC_BF16;
  int dev;
  DevInfo di;
  if (device_info(&dev, &di) != cudaSuccess) return SPEC_ERR_CUDA;
  const int epv = 16 / esz;
  p = ChainStochParams{};
  p.target = a->target_logits;
  p.draft = a->draft_logits;
  p.tokens = a->draft_tokens;
  p.temperature = a->temperature;
  p.u_accept = a->u_accept;
  p.u_sample = a->u_sample;
  p.part = static_cast<SoftPart *>(ws);
  p.B = a->B;
  p.K = K;
  p.V = a->V;
  p.use_tma = aligned(a->target_logits, 16) && (K == 0 || aligned(a->draft_logits, 16)) &&
              (static_cast<long long>(a->V) * esz) % 16 == 0;
  p.wait_limit_ns = g_wait_ns.load();
  p.force_timeout = g_force_timeout.load();
  // workspace tail: a 16-byte header {claim counter, generation, -}
  {
    char *end = static_cast<char *>(ws) + (ws_bytes & ~static_cast<size_t>(15));
    p.claim = reinterpret_cast<uint32_t *>(end - 16);
    p.gen = reinterpret_cast<uint32_t *>(end - 12);
  }
  // SPECVERIFY_DYNAMIC=0: no claimed tail in either stream kernel (tuning)
  p.stream_dyn = 1;
  if (const char *ov = std::getenv("SPECVERIFY_DYNAMIC")) p.stream_dyn = std::atoi(ov) != 0;
  {
    // the bulk-copy ring: pair tiles of 8192 bf16 / 4096 fp32 logits per law;
    // SPECVERIFY_SOFT_STAGES (2 to 4) and SPECVERIFY_DYN_CHUNK (tiles per
    // claim) override the defaults for tuning
    p.slice = kSoftThreads * kSoftVecs * epv;
    p.stages = kSoftStages;
    const char *ov = kind == StreamKind::kRing ? std::getenv("SPECVERIFY_SOFT_STAGES") : nullptr;
    if (ov) {
      const int st = std::atoi(ov);
      p.stages = st >= 2 && st <= 4 ? st : 2;
    }
    // positions 0 and 1 (where walks mostly stop) stay in L2 for the resolve
    // kernel's second look when both fit well inside it (c3: 66 MB); larger
    // batches stream every position evict-first (c5, 131 MB: 196.4 against
    // 198.6 us per step with positions 0 and 1 kept, 198.1 with position 0)
    const double pos01 = 4.0 * a->B * static_cast<double>(a->V) * esz;
    p.keep_pos = pos01 <= 0.6 * di.l2_bytes ? 2 : 0;
    if (const char *kp = std::getenv("SPECVERIFY_KEEP_POS")) p.keep_pos = std::atoi(kp);  // tuning override
    p.dyn_chunk = 2;
    if (const char *dc = std::getenv("SPECVERIFY_DYN_CHUNK")) {
      const int c = std::atoi(dc);
      if (c >= 1 && c <= 64) p.dyn_chunk = c;
    }
    p.buf_bytes = 2 * p.slice * esz;  // target tile + draft tile
    *smem = static_cast<size_t>(p.stages) * p.buf_bytes + kRingCtrlBytes;
  }
  p.nslices = ceil_div(a->V, p.slice);
  {
    const size_t rows = static_cast<size_t>(a->B) * (K + 1) + static_cast<size_t>(a->B) * K;
    p.ylog = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) +
                                                    align_up(rows * p.nslices * sizeof(SoftPart), 256));
    p.trunc = nullptr;  // set by the truncated entry point
    p.trunc_area = reinterpret_cast<SoftPart *>(reinterpret_cast<char *>(p.ylog) + align_up(rows * 8, 256));
  }
  int per_sm = 0;
  {
    if (ring_blocks(dev, bf16, p.stages, *smem, &per_sm) != cudaSuccess || per_sm < 1) return SPEC_ERR_CUDA;
    const long long tiles = static_cast<long long>(a->B) * (K + 1) * p.nslices;
    grid = static_cast<int>(std::min<long long>(tiles, static_cast<long long>(di.sms) * per_sm));
  }
  // resolve kernel: a cluster of C CTAs per row, at most 16 rounds of 32
  // vectors per warp
  constexpr int kRW = kResolveThreads / 32;
  auto rounds = [&](int c) {
    const int L = static_cast<int>(align_up(static_cast<size_t>(ceil_div(a->V, c)), static_cast<size_t>(epv)));
    return ceil_div(ceil_div(ceil_div(L, epv), kRW), 32);
  };
  C = 1;
  while (C < 16 && rounds(C) > kResolveMaxRounds) C *= 2;
  if (rounds(C) > kResolveMaxRounds) return SPEC_ERR_SHAPE;
  const int c_min = C;
  // spread each row's work over up to 8 CTAs while the whole grid stays
  // within one wave of resolve CTAs (c3: 8; B = 256: the minimum, 4)
  const long long wave = static_cast<long long>(di.sms) * kResolveBlocksPerSm;
  while (C < 8 && ceil_div(a->V, 2 * C) >= 2048 && static_cast<long long>(a->B) * 2 * C <= wave) C *= 2;
  if (const char *ov = std::getenv("SPECVERIFY_CLUSTER")) {  // tuning override
    const int c = std::atoi(ov);
    if (c >= c_min && c <= 16 && (c & (c - 1)) == 0) C = c;
  }
  p.L = static_cast<int>(align_up(static_cast<size_t>(ceil_div(a->V, C)), static_cast<size_t>(epv)));
  p.vpw = 32 * rounds(C);
  report("stochastic slice nslices grid per_sm cluster L", p.slice, p.nslices, grid, per_sm, C, p.L, 0);
  return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_verify_chain_workspace_size(int32_t B, int32_t K, int32_t V) {
  if (!valid_sizes(B, V) || K < 0 || K > SPEC_MAX_K) return 0;
  // stochastic: one partial per (logit row, slice), the smallest slice being
  // the fp32 one; greedy: one partial per (position, slice)
  const size_t rows = static_cast<size_t>(B) * (K + 1) + static_cast<size_t>(B) * K;
  const size_t soft = rows * ceil_div(V, kRecordSlice) * sizeof(SoftPart) + align_up(rows * 8, 256) +
                      rows * sizeof(SoftPart);
  const size_t part = greedy_partials_max(B, K + 1, V);
  return align_up(std::max(std::max(soft, part), static_cast<size_t>(256)), 256) + ws_tail_bytes(B);
}

size_t spec_verify_chain_truncated_workspace_size(int32_t B, int32_t K, int32_t V) {
  if (!valid_sizes(B, V) || K < 0 || K > SPEC_MAX_K) return 0;
  // the records (every area 256-byte aligned, as setup_stochastic lays them
  // out), then the chunk maxima and the kept lists
  const size_t rows = static_cast<size_t>(B) * (K + 1) + static_cast<size_t>(B) * K;
  const size_t records = align_up(rows * ceil_div(V, kRecordSlice) * sizeof(SoftPart), 256) +
                         align_up(rows * 8, 256) + align_up(rows * sizeof(SoftPart), 256);
  const size_t lists = align_up(static_cast<size_t>(B) * (K + 1) * kKeptMax * 8, 256);
  return std::max(records + chunk_max_bytes(rows, V) + lists + ws_tail_bytes(B),
                  spec_verify_chain_workspace_size(B, K, V));
}

size_t spec_verify_tree_workspace_size(int32_t B, int32_t N, int32_t V) {
  if (!valid_sizes(B, V) || N < 1 || N > SPEC_MAX_TREE_NODES) return 0;
  // the tail is reserved (unused here) so a workspace shared with chain calls
  // keeps their header
  return align_up(std::max(greedy_partials_max(B, N, V), static_cast<size_t>(256)), 256) +
         ws_tail_bytes(B);
}

spec_status spec_verify_chain(const spec_chain_args *a, const spec_chain_out *o, void *ws,
                              size_t ws_bytes, void *stream) {
  if (!a || !o) return SPEC_ERR_NULL;
  if (!valid_sizes(a->B, a->V) || a->K < 0 || a->K > SPEC_MAX_K) return SPEC_ERR_SHAPE;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (a->mode != SPEC_STOCHASTIC && a->mode != SPEC_GREEDY) return SPEC_ERR_DTYPE;
  if (std::isnan(a->margin_kappa)) return SPEC_ERR_ARG;
  if (a->B == 0) return SPEC_OK;  // nothing to do; empty arrays may be NULL
  const bool stoch = a->mode == SPEC_STOCHASTIC;
  const int K = a->K;
  if (!a->target_logits || !o->accepted_len || !o->out_tokens || !o->num_emitted ||
      !o->row_status)
    return SPEC_ERR_NULL;
  if (K > 0 && !a->draft_tokens) return SPEC_ERR_NULL;
  if (stoch && (!a->u_sample || (K > 0 && (!a->draft_logits || !a->u_accept))))
    return SPEC_ERR_NULL;
  const int esz = a->dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(a->target_logits, esz) || (stoch && a->draft_logits && !aligned(a->draft_logits, esz)))
    return SPEC_ERR_ALIGN;
  const void *i32s[] = {a->draft_tokens, a->temperature, a->u_accept, a->u_sample,
                        o->accepted_len, o->out_tokens, o->num_emitted, o->row_status,
                        o->p_at_draft, o->q_at_draft, o->resid_mass};
  for (const void *p : i32s)
    if (p && !aligned(p, 4)) return SPEC_ERR_ALIGN;
  const size_t need = spec_verify_chain_workspace_size(a->B, K, a->V);
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return SPEC_ERR_WORKSPACE;
  if (a->B == 0) return SPEC_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = a->dtype == SPEC_BF16;

  if (!stoch) {
    GreedyParams p = {};
    p.target = a->target_logits;
    p.tokens = a->draft_tokens;
    p.parent = nullptr;
    p.temperature = a->temperature;
    p.use_margin = a->margin_kappa > 0.f;
    p.ln_kappa = p.use_margin ? std::log(static_cast<double>(a->margin_kappa)) : 0.0;
    p.tree = 0;
    p.accepted_len = o->accepted_len;
    p.out_tokens = o->out_tokens;
    p.num_emitted = o->num_emitted;
    p.row_status = o->row_status;
    p.path_nodes = nullptr;
    p.B = a->B;
    p.npos = K + 1;
    p.V = a->V;
    return run_greedy(p, bf16, esz, ws, s);
  }

  ChainStochParams p;
  int grid = 0, C = 0;
  size_t smem = 0;
  {
    const spec_status st = setup_stochastic(a, ws, ws_bytes, p, grid, C, StreamKind::kRing, &smem);
    if (st != SPEC_OK) return st;
  }
  p.accepted_len = o->accepted_len;
  p.out_tokens = o->out_tokens;
  p.num_emitted = o->num_emitted;
  p.row_status = o->row_status;
  p.p_at_draft = o->p_at_draft;
  p.q_at_draft = o->q_at_draft;
  p.resid_mass = o->resid_mass;
  if (launch_chain_stochastic(p, bf16, grid, smem, C, s) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status spec_verify_chain_truncated(const spec_chain_args *a, const spec_truncation *t,
                                        const spec_chain_out *o, void *ws, size_t ws_bytes,
                                        void *stream) {
  if (!a || !t) return SPEC_ERR_NULL;
  if (a->mode != SPEC_STOCHASTIC) return SPEC_ERR_DTYPE;
  if (!t->top_k && !t->top_p) return spec_verify_chain(a, o, ws, ws_bytes, stream);
  if (a->B > 0) {
    const void *q[] = {t->top_k, t->top_p};
    for (const void *x : q)
      if (x && !aligned(x, 4)) return SPEC_ERR_ALIGN;
  }
  if (!o) return SPEC_ERR_NULL;
  if (!valid_sizes(a->B, a->V) || a->K < 0 || a->K > SPEC_MAX_K) return SPEC_ERR_SHAPE;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (a->B == 0) return SPEC_OK;
  const int K = a->K;
  if (!a->target_logits || !o->accepted_len || !o->out_tokens || !o->num_emitted ||
      !o->row_status || !a->u_sample)
    return SPEC_ERR_NULL;
  if (K > 0 && (!a->draft_tokens || !a->draft_logits || !a->u_accept)) return SPEC_ERR_NULL;
  const int esz = a->dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(a->target_logits, esz) || (a->draft_logits && !aligned(a->draft_logits, esz)))
    return SPEC_ERR_ALIGN;
  const void *i32s[] = {a->draft_tokens, a->temperature, a->u_accept, a->u_sample,
                        o->accepted_len, o->out_tokens, o->num_emitted, o->row_status,
                        o->p_at_draft, o->q_at_draft, o->resid_mass};
  for (const void *x : i32s)
    if (x && !aligned(x, 4)) return SPEC_ERR_ALIGN;
  const size_t need = spec_verify_chain_truncated_workspace_size(a->B, K, a->V);
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return SPEC_ERR_WORKSPACE;
  if (static_cast<long long>(a->B) * (2 * K + 1) > 0x7fffffffLL) return SPEC_ERR_SHAPE;
  ChainStochParams p;
  int grid = 0, C = 0;
  size_t smem = 0;
  {
    const spec_status st = setup_stochastic(a, ws, ws_bytes, p, grid, C, StreamKind::kRingListed, &smem);
    if (st != SPEC_OK) return st;
  }
  {  // the chunk maxima, after the truncation records, then the kept lists
    const size_t rows = static_cast<size_t>(a->B) * (2 * K + 1);
    char *at = reinterpret_cast<char *>(p.trunc_area) + align_up(rows * sizeof(SoftPart), 256);
    p.cmax = reinterpret_cast<unsigned short *>(at);
    at += align_up(rows * p.nslices * kSoftThreads * 2, 256);
    p.klist = reinterpret_cast<unsigned long long *>(at);
  }
  p.accepted_len = o->accepted_len;
  p.out_tokens = o->out_tokens;
  p.num_emitted = o->num_emitted;
  p.row_status = o->row_status;
  p.p_at_draft = o->p_at_draft;
  p.q_at_draft = o->q_at_draft;
  p.resid_mass = o->resid_mass;
  p.top_k = t->top_k;
  p.top_p = t->top_p;
  p.trunc = p.trunc_area;
  report("truncated grid cluster", grid, C, 0, 0, 0, 0, 0);
  return launch_chain_truncated(p, a->dtype == SPEC_BF16, grid, smem, C,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

spec_status spec_drift_residuals(const spec_chain_args *a, int32_t m, int32_t *support,
                                 float *residual, int32_t *row_status, void *ws, size_t ws_bytes,
                                 void *stream) {
  if (!a) return SPEC_ERR_NULL;
  if (!valid_sizes(a->B, a->V) || a->K < 0 || a->K > kDriftMaxK || a->B > 65535)
    return SPEC_ERR_SHAPE;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (m < 1 || m > kDriftMaxSupport || m > a->V) return SPEC_ERR_ARG;
  if (a->B == 0 || a->K == 0) return SPEC_OK;
  if (!a->target_logits || !a->draft_logits || !support || !residual || !row_status)
    return SPEC_ERR_NULL;
  const int esz = a->dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(a->target_logits, esz) || !aligned(a->draft_logits, esz)) return SPEC_ERR_ALIGN;
  const void *i32s[] = {a->temperature, a->draft_tokens, support, residual, row_status};
  for (const void *q : i32s)
    if (q && !aligned(q, 4)) return SPEC_ERR_ALIGN;
  const size_t need = spec_verify_chain_truncated_workspace_size(a->B, a->K, a->V);
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return SPEC_ERR_WORKSPACE;
  ChainStochParams p;
  int grid = 0, C = 0;
  size_t smem = 0;
  {
    const spec_status st = setup_stochastic(a, ws, ws_bytes, p, grid, C, StreamKind::kRingListed, &smem);
    if (st != SPEC_OK) return st;
  }
  {  // the target rows' chunk maxima, after the per-position records
    const size_t rows = static_cast<size_t>(a->B) * (2 * a->K + 1);
    p.cmax = reinterpret_cast<unsigned short *>(reinterpret_cast<char *>(p.trunc_area) +
                                                align_up(rows * sizeof(SoftPart), 256));
  }
  p.row_status = row_status;
  p.drift_m = m;
  p.drift_support = support;
  p.drift_residual = residual;
  report("drift grid m", grid, m, 0, 0, 0, 0, 0);
  return launch_drift(p, a->dtype == SPEC_BF16, grid, smem, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

spec_status spec_verify_chain_static(const spec_chain_args *a, const spec_chain_out *o,
                                     void *stream) {
  if (!a || !o) return SPEC_ERR_NULL;
  const size_t need = spec_verify_chain_workspace_size(a->B, a->K, a->V);
  if (need == 0) return SPEC_ERR_SHAPE;
  if (need > SPEC_STATIC_WS_BYTES) return SPEC_ERR_STATIC_LIMIT;
  int dev;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  void *ws = nullptr;
  {
    // first call on this device: look up the buffer's address (the device is
    // current here, as the lookup requires)
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_static_ws_ptr[dev]) {
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || !ptr) return SPEC_ERR_CUDA;
      g_static_ws_ptr[dev] = ptr;
    }
    ws = g_static_ws_ptr[dev];
  }
  return spec_verify_chain(a, o, ws, SPEC_STATIC_WS_BYTES, stream);
}

spec_status spec_verify_tree(const spec_tree_args *a, const spec_tree_out *o, void *ws,
                             size_t ws_bytes, void *stream) {
  if (!a || !o) return SPEC_ERR_NULL;
  if (!valid_sizes(a->B, a->V) || a->N < 1 || a->N > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (std::isnan(a->margin_kappa)) return SPEC_ERR_ARG;
  if (a->B == 0) return SPEC_OK;
  if (!a->target_logits || !a->parent || !a->node_tokens || !o->accepted_len || !o->path_nodes ||
      !o->out_tokens || !o->num_emitted || !o->row_status)
    return SPEC_ERR_NULL;
  const int esz = a->dtype == SPEC_BF16 ? 2 : 4;
  if (!aligned(a->target_logits, esz)) return SPEC_ERR_ALIGN;
  const void *i32s[] = {a->parent, a->node_tokens, a->temperature, o->accepted_len,
                        o->path_nodes, o->out_tokens, o->num_emitted, o->row_status};
  for (const void *p : i32s)
    if (p && !aligned(p, 4)) return SPEC_ERR_ALIGN;
  const size_t need = spec_verify_tree_workspace_size(a->B, a->N, a->V);
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return SPEC_ERR_WORKSPACE;
  if (a->B == 0) return SPEC_OK;
  GreedyParams p = {};
  p.target = a->target_logits;
  p.tokens = a->node_tokens;
  p.parent = a->parent;
  p.temperature = a->temperature;
  p.use_margin = a->margin_kappa > 0.f;
  p.ln_kappa = p.use_margin ? std::log(static_cast<double>(a->margin_kappa)) : 0.0;
  p.tree = 1;
  p.accepted_len = o->accepted_len;
  p.out_tokens = o->out_tokens;
  p.num_emitted = o->num_emitted;
  p.row_status = o->row_status;
  p.path_nodes = o->path_nodes;
  p.B = a->B;
  p.npos = a->N;
  p.V = a->V;
  return run_greedy(p, a->dtype == SPEC_BF16, esz, ws, static_cast<cudaStream_t>(stream));
}

spec_status spec_rollback_lengths(int32_t B, int32_t max_emit, const int32_t *kv_len_in,
                                  const int32_t *accepted_len, const int32_t *num_emitted_in,
                                  const int32_t *out_tokens, int32_t eos_id,
                                  const int32_t *max_len, int32_t *committed_kv_len,
                                  int32_t *num_emitted_out, void *stream) {
  if (B < 0 || max_emit < 1) return SPEC_ERR_SHAPE;
  if (B == 0) return SPEC_OK;
  if (!kv_len_in || !accepted_len || !num_emitted_in || !out_tokens || !committed_kv_len ||
      !num_emitted_out)
    return SPEC_ERR_NULL;
  const void *ptrs[] = {kv_len_in, accepted_len, num_emitted_in, out_tokens, max_len,
                        committed_kv_len, num_emitted_out};
  for (const void *p : ptrs)
    if (p && !aligned(p, 4)) return SPEC_ERR_ALIGN;
  if (B == 0) return SPEC_OK;
  RollbackParams p = {B, max_emit, kv_len_in, accepted_len, num_emitted_in, out_tokens, eos_id,
                      max_len, committed_kv_len, num_emitted_out};
  return launch_rollback(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK
                                                                               : SPEC_ERR_CUDA;
}

spec_status spec_workspace_init(void *ws, size_t ws_bytes, void *stream) {
  if (!ws) return SPEC_ERR_NULL;
  return cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

const char *spec_status_string(spec_status s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_NULL: return "SPEC_ERR_NULL: a required pointer is NULL";
    case SPEC_ERR_SHAPE: return "SPEC_ERR_SHAPE: a size is outside the supported range";
    case SPEC_ERR_DTYPE: return "SPEC_ERR_DTYPE: unknown dtype or mode";
    case SPEC_ERR_ALIGN: return "SPEC_ERR_ALIGN: a pointer is misaligned";
    case SPEC_ERR_ARG: return "SPEC_ERR_ARG: bad scalar argument";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA: a CUDA runtime call failed";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SPEC_ERR_STATIC_LIMIT:
      return "SPEC_ERR_STATIC_LIMIT: the problem needs more scratch than the built-in "
             "SPEC_STATIC_WS_BYTES buffer of spec_verify_chain_static holds";
  }
  return "unknown spec_status";
}

void spec_set_wait_timeout_ns(uint64_t ns) { g_wait_ns.store(ns); }
uint64_t spec_get_wait_timeout_ns(void) { return g_wait_ns.load(); }
void spec_debug_force_wait_timeout(int on) { g_force_timeout.store(on ? 1 : 0); }

#ifdef SV_BOUNDS
// Bounds-check builds only (-DSV_BOUNDS): the number of bad indexes the
// chain and tree kernels met since the last call, and the source line of the
// first; both records are cleared.  Returns the CUDA error of the reads.
int spec_debug_bounds(unsigned *count, unsigned *line) {
  *count = 0u;
  *line = 0u;
  cudaError_t e = oob_record_chain(count, line);
  if (e == cudaSuccess) e = oob_record_greedy(count, line);
  return static_cast<int>(e);
}

// Bounds-check builds only: enqueue a check that fails by design, touching
// no memory, so that a test can see the record work.
int spec_debug_bounds_selftest(void *stream) {
  return static_cast<int>(oob_selftest(static_cast<cudaStream_t>(stream)));
}
#endif

}  // extern "C"
