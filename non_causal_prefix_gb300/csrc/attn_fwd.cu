// BF16 attention forward for GB300 (sm_103a): the host side and the C ABI of
// include/ncp_attn.h.  The kernel itself is in attn_kernel.cuh (persistent,
// warp-specialised: TMA-staged K/V tiles, tcgen05 MMAs accumulating S = Q K^T
// and O = P V in tensor memory, online softmax in registers), its PTX
// building blocks in sm103_ptx.cuh.
//
// Operations (page "Audit SGLang interfaces and refresh validated kernel
// solutions", dataset definitions, field "reference"):
//   dense:   noncausal_dense_attention_h32_d{128,64} -- softmax(Q K^T * D^-0.5) V,
//            no mask; cross attention (Nq != Nk) allowed.
//   prefix:  prefix_cached_block_causal_h32_d128 -- keys/values are
//            cat(prefix, current) on the token axis, every key visible; walked
//            as two pairs of TMA descriptors (no copy).
//   block-causal: prefix_cached_block_causal_h32_d128_prefix0 -- causal text,
//            bidirectional inside each image block.
//   masked prefix: the pre-audit form of the prefix definition (image ids over
//            prefix + current, key_valid, runtime sm_scale).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <algorithm>
#include <mutex>
#include <vector>
#include <utility>

#include "ncp_attn.h"
#include "attn_kernel.cuh"

// ============================================================================
// Fixed scratch for attn_dense_fwd_noalloc: the split workspace (arrival
// counters, then partials) of a call that may not allocate, as one static
// device array.  Every GPU that loads this library holds it until the process
// exits.  Sized for any GPU with up to 160 SMs at D <= 128: 320 counters in a
// 256-byte aligned block, then 320 partial slots of 2 x 128 x (128 + 4) floats.
// ============================================================================
namespace ncp {
constexpr int NOALLOC_SLOTS = 320;
constexpr int NOALLOC_COUNTERS = 320;
constexpr size_t NOALLOC_COUNT_BYTES = NOALLOC_COUNTERS * sizeof(unsigned long long);  // 2560
constexpr size_t NOALLOC_PART_BYTES =
    static_cast<size_t>(NOALLOC_SLOTS) * 2 * (128 + 4) * BM * sizeof(float);
constexpr size_t NOALLOC_SCRATCH_BYTES = NOALLOC_COUNT_BYTES + NOALLOC_PART_BYTES;  // 43.3 MB
static_assert(NOALLOC_COUNT_BYTES % 256 == 0, "partial rows start 256-byte aligned");
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];
}  // namespace ncp

// ============================================================================
// Host side: argument checks, TMA descriptors, launch
// ============================================================================
namespace {

using ncp::Params;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

std::mutex g_cfg_mutex;
int g_fault_mode = 0;
unsigned long long g_wait_limit_ns = 2000000000ull;

// [B, N, H, D] bf16, box of 64 head-dim elements x 1 head x 128 tokens x 1
// batch, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* map, const void* base, int B, int N, int H, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(N) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// ---------------------------------------------------------------------------
// Work schedule (see ncp::schedule_item): whole units fill complete rounds of
// one persistent CTA per SM.  When the units left for a last, partly filled
// round would leave SMs idle, their key tiles are shared out evenly over the
// CTAs instead, each unit's pieces merged through a workspace.
// ---------------------------------------------------------------------------
// Schedule of n_units units of (at most) T key tiles each on `sms` SMs;
// `can_split` false (no workspace) keeps every unit whole.  The masked forms
// visit a data-dependent subset of each unit's key tiles: T bounds their
// work here, and the kernel shares out the tail by the tiles actually
// visited.  Returns the grid size.
// Cost of one extra tail piece on a CTA, in key-tile times: its Q load and
// pipeline fill, its partial written and counted in, and the merge.  On
// GB300 a CTA with two tail pieces ends about 6 tiles after one with a single
// piece of the same length, but part of that overlaps.  Of the costs 1, 2, 3,
// 5 and 8 tried, 3 gave the shortest launches.  (Re-measured with 2, 3, 4 and
// 6: 4 was up to 1.6 % faster on the split workloads, but on short key
// sequences it stops splitting tails that 3 still splits.)
#ifndef NCP_PIECE_COST
#define NCP_PIECE_COST 3
#endif
constexpr long long PIECE_COST = NCP_PIECE_COST;

// Dense tail ranges: cut W tail tiles (units of T tiles, in order) into
// consecutive non-empty ranges, each CTA's tiles plus PIECE_COST for every
// unit boundary it crosses at most `cap`; a CTA only crosses into the next
// unit with budget left for a tile there.  Returns the number of ranges
// (bounds[0 .. n]), or -1 if more than g are needed.
int tail_ranges(long long W, long long T, long long g, long long cap, int* bounds) {
  long long pos = 0;
  int n = 0;
  bounds[0] = 0;
  while (pos < W) {
    if (n >= g) return -1;
    long long budget = cap;
    while (true) {
      const long long take = std::min(T - pos % T, std::min(budget, W - pos));
      pos += take;
      budget -= take;
      if (pos >= W || budget <= PIECE_COST || pos % T != 0) break;
      budget -= PIECE_COST;  // cross into the next unit
    }
    bounds[++n] = static_cast<int>(pos);
  }
  return n;
}

// Dense units of at most this many key tiles are short enough that their
// item boundaries, where the next Q loads from HBM, weigh: the loader then
// prefetches each next Q into L2 (Sched::prefetch_q; D = 128 kernel only).
// Measured on cross Nq=8192 Nk=512: 67.2 -> 64.2 us.  On longer key
// sequences the prefetch measured no faster.
constexpr int PREFETCH_Q_MAX_TILES = 8;

int make_sched(ncp::Sched& s, long long n_units, int T, int sms, bool can_split, bool masked) {
  s.n_units = static_cast<int>(n_units);
  s.n_whole = s.n_units;
  s.tail_units = 0;
  s.tail_ctas = 0;
  s.prefetch_q = (!masked && T <= PREFETCH_Q_MAX_TILES) ? 1 : 0;
  const long long rem = n_units % sms;
  if (can_split && rem > 0) {
    const long long W = rem * T;
    long long g_tail = sms;
    if (g_tail > W / ncp::MIN_PIECE_TILES) g_tail = W / ncp::MIN_PIECE_TILES;
    if (g_tail > rem * ncp::MAX_PIECES) g_tail = rem * ncp::MAX_PIECES;
    if (!masked && g_tail > ncp::MAX_TAIL_CTAS) g_tail = ncp::MAX_TAIL_CTAS;
    if (g_tail > rem && rem <= ncp::MAX_TAIL_UNITS) {
      s.n_whole = static_cast<int>(n_units - rem);
      s.tail_units = static_cast<int>(rem);
      s.tail_ctas = static_cast<int>(g_tail);
      if (!masked) {
        // The least per-CTA cost whose ranges fit in g_tail CTAs (binary
        // search; one CTA taking everything always fits).
        long long lo = (W + g_tail - 1) / g_tail, hi = W + PIECE_COST * rem;
        while (lo < hi) {
          const long long mid = (lo + hi) / 2;
          if (tail_ranges(W, T, g_tail, mid, s.bounds) >= 0) hi = mid; else lo = mid + 1;
        }
        s.tail_ctas = tail_ranges(W, T, g_tail, lo, s.bounds);
      }
      return s.n_whole > 0 ? sms : s.tail_ctas;
    }
  }
  return n_units < sms ? static_cast<int>(n_units) : sms;
}

// Workspace slots a schedule uses: tail piece (CTA c, tail unit r) takes slot
// c + r, so fewer than tail_ctas + tail_units (< 2 x SMs).
int sched_slots(const ncp::Sched& s) { return s.tail_ctas ? s.tail_ctas + s.tail_units - 1 : 0; }

// Bytes of partials for `slots` pieces: 2 query tiles x 128 rows x (128 + 4)
// floats (O, then m and l, at D <= 128).
size_t part_bytes(long long slots) {
  return static_cast<size_t>(slots) * 2 * (128 + 4) * ncp::BM * sizeof(float);
}

// ---------------------------------------------------------------------------
// Split workspaces: partials of the tail pieces (2 x SMs slots) plus one
// arrival counter per (tail unit, query tile).  A bounded pool per device:
// at most WS_PER_DEVICE of them, each created by the first call that needs
// it (cudaMalloc) and kept until the process exits.  A call takes, in this
// order:
//   1. the workspace its stream used last;
//   2. a workspace no other stream has work pending on (its completion
//      event has fired) and that no graph capture has claimed;
//   3. a new one, while the pool has room;
// and otherwise runs without splitting.  The call enqueues a wait on the
// workspace's completion event (nothing, if it has fired), launches, and
// records the event again; the pool lock is held throughout, so two calls
// never take one workspace at once.  Calls that run concurrently on
// different streams therefore never share a workspace, and the device memory
// the pool holds is bounded whatever streams come and go.
//
// Each launch tags its arrival counters with a fresh epoch (see
// Params::epoch): a launch that gave up part-way leaves counters that the
// next one ignores.  A call made while its stream is being captured into a
// graph uses only a workspace that stream used last, claims it for good (no
// other stream takes it afterwards) and clears its counters in a captured
// memset before the kernel, because every replay repeats the captured epoch.
// Without such a workspace a captured call runs unsplit: nothing is
// allocated, queried or awaited during a capture.
// ---------------------------------------------------------------------------
constexpr int WS_PER_DEVICE = 4;

struct Workspace {
  float* part = nullptr;
  unsigned long long* count = nullptr;
  size_t count_bytes = 0;
  cudaEvent_t done = nullptr;  // recorded after each launch that used it
  uintptr_t last_stream = 0;   // stream handle of the last launch that used it
  bool claimed = false;        // used by a captured graph: only last_stream may take it
  unsigned int epoch = 0;      // tag of the last launch (0: none yet)
};

std::mutex g_ws_mutex;
std::vector<Workspace*> g_ws[64];  // per device, never shrinks below what it made

unsigned int next_epoch(Workspace& ws) {
  if (++ws.epoch == 0) ws.epoch = 1;  // 0 is a cleared counter's tag
  return ws.epoch;
}

// A new workspace on the current device, its counters cleared on `stream`,
// or nullptr if allocation fails.
Workspace* new_workspace(int sms, cudaStream_t stream) {
  Workspace* ws = new Workspace;
  ws->count_bytes = static_cast<size_t>(2) * sms * sizeof(unsigned long long);
  if (cudaMalloc(reinterpret_cast<void**>(&ws->part), part_bytes(2LL * sms)) != cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&ws->count), ws->count_bytes) != cudaSuccess ||
      cudaMemsetAsync(ws->count, 0, ws->count_bytes, stream) != cudaSuccess ||
      cudaEventCreateWithFlags(&ws->done, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    if (ws->part) cudaFree(ws->part);
    if (ws->count) cudaFree(ws->count);
    delete ws;
    return nullptr;
  }
  return ws;
}

// Picks this call's workspace from the device's pool (see above) and enqueues
// what must come before the kernel on `stream`.  Called with g_ws_mutex held;
// returns nullptr when the call must run unsplit.
Workspace* take_workspace(int dev, int sms, cudaStream_t stream, bool capturing) {
  std::vector<Workspace*>& pool = g_ws[dev];
  const uintptr_t key = reinterpret_cast<uintptr_t>(stream);
  Workspace* pick = nullptr;
  for (Workspace* ws : pool)
    if (ws->last_stream == key) { pick = ws; break; }
  if (capturing) {
    if (!pick) return nullptr;
    if (cudaMemsetAsync(pick->count, 0, pick->count_bytes, stream) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    pick->claimed = true;
    return pick;
  }
  if (!pick) {
    for (Workspace* ws : pool) {
      if (ws->claimed) continue;
      const cudaError_t q = cudaEventQuery(ws->done);
      if (q == cudaSuccess) { pick = ws; break; }
      if (q != cudaErrorNotReady) cudaGetLastError();
    }
  }
  if (!pick && static_cast<int>(pool.size()) < WS_PER_DEVICE) {
    pick = new_workspace(sms, stream);
    if (pick) pool.push_back(pick);
  }
  if (!pick) return nullptr;
  // Stream-ordered after the workspace's previous launch (a no-op when that
  // was on this stream, or has finished).
  if (cudaStreamWaitEvent(stream, pick->done, 0) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return pick;
}

// SM count of the current device, with the kernel's shared-memory limit set
// there (once per device and instantiation).
template <int D, bool BC>
int configure(int* dev_out, int* sms_out) {
  using C = ncp::Cfg<D>;
  constexpr uint32_t smem = BC ? C::SMEM_BYTES_BC : C::SMEM_BYTES;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  static int sm_count[64] = {};  // per device, 0 = not configured yet
  if (dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  if (sm_count[dev] == 0) {
    int sms = 0;
    if (cudaFuncSetAttribute(ncp::attn_fwd_kernel<D, BC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1)
      return ATTN_ERR_CUDA;
    sm_count[dev] = sms;
  }
  *dev_out = dev;
  *sms_out = sm_count[dev];
  return ATTN_OK;
}

template <int D, bool BC>
int launch(Params& prm, long long n_units, cudaStream_t stream) {
  using C = ncp::Cfg<D>;
  constexpr uint32_t smem = BC ? C::SMEM_BYTES_BC : C::SMEM_BYTES;
  int dev = 0, sms = 0;
  if (configure<D, BC>(&dev, &sms) != ATTN_OK) return ATTN_ERR_CUDA;
  const int T = prm.n_tiles[0] + prm.n_tiles[1];
  int grid = make_sched(prm.sc, n_units, T, sms, true, BC);
  prm.ws_part = nullptr;
  prm.ws_count = nullptr;
  prm.epoch = 1;
  if (prm.sc.tail_ctas == 0) {
    ncp::attn_fwd_kernel<D, BC><<<grid, ncp::num_threads<D>(), smem, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  Workspace* ws = take_workspace(dev, sms, stream, capturing);
  if (!ws) {
    grid = make_sched(prm.sc, n_units, T, sms, false, BC);
    ncp::attn_fwd_kernel<D, BC><<<grid, ncp::num_threads<D>(), smem, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  prm.ws_part = ws->part;
  prm.ws_count = ws->count;
  prm.epoch = next_epoch(*ws);
  ncp::attn_fwd_kernel<D, BC><<<grid, ncp::num_threads<D>(), smem, stream>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  ws->last_stream = reinterpret_cast<uintptr_t>(stream);
  if (!capturing && cudaEventRecord(ws->done, stream) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// Argument checks, TMA descriptors and kernel parameters of one call.
int prepare(const void* q, const void* kp, const void* vp, const void* kc, const void* vc,
            const int* image_ids, const unsigned char* key_valid, float sm_scale, void* out, int B,
            int Nq, int Np, int Nc, int H, int D, Params& prm, long long& n_units) {
  if (!q || !kc || !vc || !out || (Np > 0 && (!kp || !vp))) return ATTN_ERR_NULL;
  if (B < 1 || Nq < 1 || Nc < 1 || H < 1 || Np < 0) return ATTN_ERR_SHAPE;
  if (H > 65535 || B > 65535) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  if (misaligned(q) || misaligned(kc) || misaligned(vc) || misaligned(out) ||
      (Np > 0 && (misaligned(kp) || misaligned(vp))))
    return ATTN_ERR_ALIGN;
  const size_t row = static_cast<size_t>(H) * D * 2;
  const size_t q_bytes = static_cast<size_t>(B) * Nq * row;
  const size_t c_bytes = static_cast<size_t>(B) * Nc * row;
  const size_t p_bytes = static_cast<size_t>(B) * Np * row;
  if (overlaps(out, q_bytes, q, q_bytes) || overlaps(out, q_bytes, kc, c_bytes) ||
      overlaps(out, q_bytes, vc, c_bytes) ||
      (Np > 0 && (overlaps(out, q_bytes, kp, p_bytes) || overlaps(out, q_bytes, vp, p_bytes))))
    return ATTN_ERR_ALIAS;

  if (!make_map(&prm.tm_q, q, B, Nq, H, D)) return ATTN_ERR_CUDA;
  if (!make_map(&prm.tm_k[1], kc, B, Nc, H, D) || !make_map(&prm.tm_v[1], vc, B, Nc, H, D))
    return ATTN_ERR_CUDA;
  if (Np > 0) {
    if (!make_map(&prm.tm_k[0], kp, B, Np, H, D) || !make_map(&prm.tm_v[0], vp, B, Np, H, D))
      return ATTN_ERR_CUDA;
  } else {
    prm.tm_k[0] = prm.tm_k[1];
    prm.tm_v[0] = prm.tm_v[1];
  }
  const long long q_pairs = (static_cast<long long>(Nq) + 2 * ncp::BM - 1) / (2 * ncp::BM);
  n_units = static_cast<long long>(B) * H * q_pairs;
  if (n_units > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.image_ids = image_ids;
  prm.key_valid = key_valid;
  prm.Nq = Nq;
  prm.H = H;
  prm.sc.n_units = static_cast<int>(n_units);
  prm.sc.q_pairs = static_cast<int>(q_pairs);
  prm.sc.H = H;
  prm.sc.Nq = Nq;
  prm.sc.unit_rows = 2 * ncp::BM;
  prm.n_tok[0] = Np;
  prm.n_tok[1] = Nc;
  prm.n_tiles[0] = (Np + ncp::BN - 1) / ncp::BN;
  prm.n_tiles[1] = (Nc + ncp::BN - 1) / ncp::BN;
  // Scale D^-0.5 unless the call passes one (sm_scale > 0), times log2(e).
  const double scale = sm_scale > 0.f ? static_cast<double>(sm_scale)
                                      : 1.0 / std::sqrt(static_cast<double>(D));
  prm.scale_log2 = static_cast<float>(1.4426950408889634 * scale);
  {
    std::lock_guard<std::mutex> lock(g_cfg_mutex);
    prm.fault_mode = g_fault_mode;
    prm.wait_limit_ns = g_wait_limit_ns;
  }
  return ATTN_OK;
}

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (in host code the array's name is only a host-side stand-in).
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[64] = {};

int noalloc_scratch(int dev, void** addr) {
  if (dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, ncp::g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_noalloc_addr[dev] = ptr;
  }
  *addr = g_noalloc_addr[dev];
  return ATTN_OK;
}

// The schedule of launch<D> with the split workspace taken from the static
// scratch: no allocation.  A schedule that would need more slots than the
// scratch holds is refused (ATTN_ERR_SHAPE); the counters are cleared on the
// stream first, since an aborted earlier call may have left them non-zero.
template <int D>
int launch_noalloc(Params& prm, long long n_units, cudaStream_t stream) {
  using C = ncp::Cfg<D>;
  int dev = 0, sms = 0;
  if (configure<D, false>(&dev, &sms) != ATTN_OK) return ATTN_ERR_CUDA;
  const int T = prm.n_tiles[0] + prm.n_tiles[1];
  const int grid = make_sched(prm.sc, n_units, T, sms, true, false);
  if (sched_slots(prm.sc) > ncp::NOALLOC_SLOTS || 2 * prm.sc.tail_units > ncp::NOALLOC_COUNTERS)
    return ATTN_ERR_SHAPE;
  void* scratch = nullptr;
  if (noalloc_scratch(dev, &scratch) != ATTN_OK) return ATTN_ERR_CUDA;
  if (prm.sc.tail_ctas > 0 &&
      cudaMemsetAsync(scratch, 0, ncp::NOALLOC_COUNT_BYTES, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  prm.ws_count = static_cast<unsigned long long*>(scratch);
  prm.epoch = 1;  // the counters were just cleared (tag 0)
  prm.ws_part = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) +
                                         ncp::NOALLOC_COUNT_BYTES);
  ncp::attn_fwd_kernel<D, false><<<grid, ncp::num_threads<D>(), C::SMEM_BYTES, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int run(const void* q, const void* kp, const void* vp, const void* kc, const void* vc,
        const int* image_ids, const unsigned char* key_valid, float sm_scale, void* out, int B,
        int Nq, int Np, int Nc, int H, int D, cudaStream_t stream) {
  Params prm;
  long long n_units = 0;
  const int rc = prepare(q, kp, vp, kc, vc, image_ids, key_valid, sm_scale, out, B, Nq, Np, Nc, H,
                         D, prm, n_units);
  if (rc != ATTN_OK) return rc;
  if (image_ids)
    return D == 128 ? launch<128, true>(prm, n_units, stream)
                    : launch<64, true>(prm, n_units, stream);
  return D == 128 ? launch<128, false>(prm, n_units, stream)
                  : launch<64, false>(prm, n_units, stream);
}

}  // namespace

extern "C" {

int attn_dense_fwd(const void* q, const void* k, const void* v, void* out, int B, int N, int H,
                   int D, cudaStream_t stream) {
  if (!k || !v) return ATTN_ERR_NULL;
  return run(q, nullptr, nullptr, k, v, nullptr, nullptr, 0.f, out, B, N, 0, N, H, D, stream);
}

int attn_dense_cross_fwd(const void* q, const void* k, const void* v, void* out, int B, int Nq,
                         int Nk, int H, int D, cudaStream_t stream) {
  if (!k || !v) return ATTN_ERR_NULL;
  return run(q, nullptr, nullptr, k, v, nullptr, nullptr, 0.f, out, B, Nq, 0, Nk, H, D, stream);
}

int attn_masked_prefix_fwd(const void* q, const void* kc, const void* vc, const void* kp,
                           const void* vp, const int* image_ids, const unsigned char* key_valid,
                           float sm_scale, void* out, int B, int Nq, int Np, int H, int D,
                           cudaStream_t stream) {
  if (!kc || !vc || !image_ids) return ATTN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(image_ids) & 15u) != 0) return ATTN_ERR_ALIGN;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return ATTN_ERR_SHAPE;
  if (Np < 0 || Nq < 1 || static_cast<long long>(Np) + Nq > ncp::MAX_SEQ_TILES * ncp::BN ||
      (Np + ncp::BN - 1) / ncp::BN + (Nq + ncp::BN - 1) / ncp::BN > ncp::MAX_SEQ_TILES)
    return ATTN_ERR_SHAPE;
  const size_t n_all = static_cast<size_t>(Np) + Nq;
  if (B >= 1 && H >= 1 && D >= 1) {
    const size_t o_bytes = static_cast<size_t>(B) * Nq * H * D * 2;
    if (overlaps(out, o_bytes, image_ids, n_all * sizeof(int)) ||
        (key_valid && overlaps(out, o_bytes, key_valid, static_cast<size_t>(B) * n_all)))
      return ATTN_ERR_ALIAS;
  }
  return run(q, kp, vp, kc, vc, image_ids, key_valid, sm_scale, out, B, Nq, Np, Nq, H, D, stream);
}

int attn_block_causal_fwd(const void* q, const void* k, const void* v, const int* image_ids,
                          void* out, int B, int N, int H, int D, cudaStream_t stream) {
  if (!k || !v || !image_ids) return ATTN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(image_ids) & 15u) != 0) return ATTN_ERR_ALIGN;
  if (N > ncp::MAX_SEQ_TILES * ncp::BN) return ATTN_ERR_SHAPE;
  if (B >= 1 && N >= 1 && H >= 1 && D >= 1 &&
      overlaps(out, static_cast<size_t>(B) * N * H * D * 2, image_ids,
               static_cast<size_t>(N) * sizeof(int)))
    return ATTN_ERR_ALIAS;
  return run(q, nullptr, nullptr, k, v, image_ids, nullptr, 0.f, out, B, N, 0, N, H, D, stream);
}

int attn_dense_fwd_noalloc(const void* q, const void* k, const void* v, void* out, int B, int N,
                           int H, int D, cudaStream_t stream) {
  if (!k || !v) return ATTN_ERR_NULL;
  Params prm;
  long long n_units = 0;
  const int rc =
      prepare(q, nullptr, nullptr, k, v, nullptr, nullptr, 0.f, out, B, N, 0, N, H, D, prm, n_units);
  if (rc != ATTN_OK) return rc;
  return D == 128 ? launch_noalloc<128>(prm, n_units, stream)
                  : launch_noalloc<64>(prm, n_units, stream);
}

int attn_prefix_fwd(const void* q, const void* kp, const void* vp, const void* kc, const void* vc,
                    void* out, int B, int Nq, int Np, int Nc, int H, int D, cudaStream_t stream) {
  return run(q, kp, vp, kc, vc, nullptr, nullptr, 0.f, out, B, Nq, Np, Nc, H, D, stream);
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "null pointer";
    case ATTN_ERR_SHAPE: return "size out of range";
    case ATTN_ERR_HEADDIM: return "head dim must be 64 or 128";
    case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
    case ATTN_ERR_ALIAS: return "output overlaps an input";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "in-kernel wait timed out";
    default: return "unknown status";
  }
}

int attn_device_status(cudaStream_t stream, unsigned int* info) {
  if (info) *info = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int st = 0, inf = 0;
  if (cudaMemcpyFromSymbol(&st, ncp::g_status, sizeof st) != cudaSuccess) return ATTN_ERR_CUDA;
  if (st == 0) return ATTN_OK;
  if (cudaMemcpyFromSymbol(&inf, ncp::g_status_info, sizeof inf) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(ncp::g_status, &zero, sizeof zero) != cudaSuccess ||
      cudaMemcpyToSymbol(ncp::g_status_info, &zero, sizeof zero) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (info) *info = inf;
  return ATTN_ERR_TIMEOUT;
}

int attn_debug_exp2(const float* x, float* y, long long n, int mode, cudaStream_t stream) {
  if (n < 0 || (mode != 0 && mode != 1)) return ATTN_ERR_SHAPE;
  if (n == 0) return ATTN_OK;
  if (!x || !y) return ATTN_ERR_NULL;
  const long long pairs = (n + 1) / 2;
  const long long blocks = (pairs + 255) / 256;
  if (blocks > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  ncp::exp2_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, y, n, mode);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_debug_schedule(int B, int Nq, int H, int n_key_tiles, int sms, int masked,
                        const int* image_ids, int Np, int* rows, int cap, int* n_rows,
                        int* grid_out, int* slots_out) {
  if (!n_rows || !grid_out || !slots_out || (cap > 0 && !rows)) return ATTN_ERR_NULL;
  if (B < 1 || Nq < 1 || H < 1 || sms < 1 || cap < 0 || Np < 0 || masked < 0 || masked > 1)
    return ATTN_ERR_SHAPE;
  const int unit_rows = 2 * ncp::BM;
  ncp::Params prm{};
  prm.Nq = Nq;
  prm.H = H;
  prm.n_tok[0] = masked ? Np : 0;
  prm.n_tok[1] = Nq;
  prm.n_tiles[0] = masked ? (Np + ncp::BN - 1) / ncp::BN : 0;
  prm.n_tiles[1] = masked ? (Nq + ncp::BN - 1) / ncp::BN : n_key_tiles;
  const int T = prm.n_tiles[0] + prm.n_tiles[1];
  if (T < 1 || (masked && T > ncp::MAX_SEQ_TILES)) return ATTN_ERR_SHAPE;
  const long long q_pairs = (static_cast<long long>(Nq) + unit_rows - 1) / unit_rows;
  const long long n_units = static_cast<long long>(B) * H * q_pairs;
  if (n_units > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  ncp::Sched& s = prm.sc;
  s.q_pairs = static_cast<int>(q_pairs);
  s.H = H;
  s.Nq = Nq;
  s.unit_rows = unit_rows;
  const int grid = make_sched(s, n_units, T, sms, true, masked != 0);
  // Masked forms: the kernel's tile table and tail prefix sums, built here.
  std::vector<int> table(3 * ncp::MAX_SEQ_TILES, 0), pre(s.tail_units + 1, 0);
  std::vector<int> order(ncp::ORDER_QP + 2 * ncp::MAX_Q_PAIRS, 0);
  ncp::MaskedTail mt{&prm, ncp::TileTable{table.data()}, pre.data(), nullptr, 0,
                     ncp::UnitOrder{order.data()}};
  if (masked) {
    if (!image_ids) return ATTN_ERR_NULL;
    if (q_pairs > ncp::MAX_Q_PAIRS) return ATTN_ERR_SHAPE;
    for (int t = 0; t < T; ++t)
      ncp::tile_summary(prm, image_ids, t, table[t], table[ncp::MAX_SEQ_TILES + t],
                        table[2 * ncp::MAX_SEQ_TILES + t]);
    int* cnt = order.data() + ncp::ORDER_QP + ncp::MAX_Q_PAIRS;
    for (int q = 0; q < s.q_pairs; ++q) {
      ncp::Unit uq{0, 0, q * 2 * ncp::BM, q * 2 * ncp::BM + ncp::BM < Nq};
      for (int t = 0; t < T; ++t) cnt[q] += ncp::bc_pair_tile_cost(mt.tt, prm, uq, t);
    }
    for (int q = 0; q < s.q_pairs; ++q)
      order[ncp::ORDER_QP + ncp::order_rank(cnt, s.q_pairs, q)] = q;
    ncp::order_levels(order.data(), cnt, s.q_pairs);
    for (int r = 0; r < s.tail_units; ++r) {
      const ncp::Unit u = ncp::decode_unit(s, true, s.n_whole + r, &mt.ord);
      int cnt = 0;
      for (int t = 0; t < T; ++t) cnt += ncp::bc_unit_visits(mt.tt, prm, u, t) ? 1 : 0;
      pre[r + 1] = pre[r] + cnt;
    }
  }
  long long count = 0;
  ncp::Item it;
  for (int c = 0; c < grid; ++c)
    for (int n = 0; masked ? ncp::schedule_item<true>(s, T, grid, c, n, it, &mt)
                           : ncp::schedule_item<false>(s, T, grid, c, n, it, nullptr);
         ++n, ++count) {
      if (count >= cap) continue;
      int* r = rows + 12 * count;
      const int v[12] = {c, n, it.u.b, it.u.h, it.u.q0, it.u.two ? 1 : 0, it.t_begin, it.t_end,
                         it.tail, it.piece, it.pieces, it.slot0};
      for (int e = 0; e < 12; ++e) r[e] = v[e];
    }
  *n_rows = static_cast<int>(count < 0x7fffffffLL ? count : 0x7fffffffLL);
  *grid_out = grid;
  *slots_out = sched_slots(s);
  return count <= cap ? ATTN_OK : ATTN_ERR_SHAPE;
}

int attn_debug_set_fault(int mode, unsigned int wait_limit_us) {
  if (mode < 0 || mode > 1) return ATTN_ERR_SHAPE;
  std::lock_guard<std::mutex> lock(g_cfg_mutex);
  g_fault_mode = mode;
  g_wait_limit_ns = wait_limit_us ? static_cast<unsigned long long>(wait_limit_us) * 1000ull
                                  : 2000000000ull;
  return ATTN_OK;
}

}  // extern "C"
