// sr_api.cu -- the C ABI of libsr.so (declared in include/sr.h): argument
// validation, the per-session state machine, tensor-map encoding and launches.
//
// Host state per session mirrors the streaming loop of the H3 project page
// ("Interactive Coding Worlds with Real-time Streaming Diffusion Render"):
// static-context banks written once (section 3.3 "Static-context KV caching"),
// a preallocated ring of W frames updated in place (section 3.2 Iteration 3
// item 2; 3.3 "Persistent KV layout") and the number of frames committed so
// far, which fixes both the rotary time of the chunk and the occupied ring
// prefix. Everything an attention call needs is derived on the host from that
// count, so no call waits on the device (section 3.3 "Attention metadata
// reuse": no host-device synchronisation per call).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>
#include <queue>
#include <vector>

#include "sr.h"
#include "sr_kernels.h"

struct sr_session {
  sr_config cfg;
  sr_buffers buf;
  int64_t tokens_per_frame;   // T
  int64_t lq;                 // F*T
  float scale;
  int64_t n_committed;
  int32_t epoch;              // attention calls so far (key-split counters)
  bool counters_stale;        // the epoch wrapped: clear the workspace counters before the next launch
  int64_t plan_key[4];        // the launch plan last chosen (choose_plan), and what it was chosen for
  int32_t plan_split, plan_conv;
  sr::RopePhase phase;        // per rotary pair: axis and fixed-point turn constant
  // Tensor maps encoded for this session's calls, by (address, rows): a map
  // holds only the address, extents and strides, so a buffer that comes back
  // (the banks, the ring, a caller's reused chunk buffers) reuses its map.
  struct MapEntry {
    const void* base;
    int64_t rows;
    CUtensorMap map;
  } maps[16];
  int32_t map_next;
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// The slot table holds absolute frame indices as int32: a session commits at
// most this many frames.
constexpr int64_t kMaxFrames = INT32_MAX;
constexpr int kBoxRows = 128;
constexpr int kBoxCols = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sr_status validate_config(const sr_config& c) {
  if (c.n_heads < 1 || c.grid_h < 1 || c.grid_w < 1 || c.chunk_frames < 1 || c.window_frames < 0 ||
      c.n_sink < 0 || c.n_steps < 1)
    return SR_ERR_INVALID_ARG;
  if (c.head_dim != 64 && c.head_dim != 128) return SR_ERR_UNSUPPORTED;
  if (c.window_frames > 0 && c.window_frames < c.chunk_frames) return SR_ERR_INVALID_ARG;
  if (!(c.rope_base > 1.0f) || !std::isfinite(c.rope_base)) return SR_ERR_INVALID_ARG;
  if (!std::isfinite(c.softmax_scale)) return SR_ERR_INVALID_ARG;
  if (c.tail_split < 0 || c.tail_split > SR_MAX_TAIL_SPLIT) return SR_ERR_INVALID_ARG;
  // every element offset must fit comfortably in 32-bit row counts
  const int64_t row = static_cast<int64_t>(c.n_heads) * c.head_dim;
  const int64_t T = static_cast<int64_t>(c.grid_h) * c.grid_w;
  const int64_t lq = T * c.chunk_frames;
  const int64_t ring_rows = T * c.window_frames;
  const int64_t limit = int64_t(1) << 30;
  if (row > 65536 || lq > limit / 4 || ring_rows > limit / 4 || c.n_sink > limit / 4 ||
      lq * row > limit || ring_rows * row > limit || static_cast<int64_t>(c.n_sink) * row * c.n_steps > limit)
    return SR_ERR_INVALID_ARG;
  return SR_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D map over a token-major bf16 tensor [rows][row_elems], box {64, 128},
// 128-byte swizzle, zero fill outside [0, rows).
bool encode_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t row_elems) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_elems), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems * 2)};
  cuuint32_t box[2] = {kBoxCols, kBoxRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// encode_rows through the session's map cache (s may be NULL: no cache).
bool encode_cached(sr_session* s, CUtensorMap* map, const void* base, int64_t rows, int64_t row_elems) {
  if (s == nullptr) return encode_rows(map, base, rows, row_elems);
  for (const auto& e : s->maps)
    if (e.base == base && e.rows == rows && base != nullptr) {
      *map = e.map;
      return true;
    }
  if (!encode_rows(map, base, rows, row_elems)) return false;
  auto& e = s->maps[s->map_next];
  s->map_next = (s->map_next + 1) % 16;
  e.base = base;
  e.rows = rows;
  e.map = *map;
  return true;
}

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

// Max dynamic shared memory is a per-device function attribute: set it once
// per device and template.
cudaError_t ensure_attn_attr(int head_dim, int nsess_template) {
  static std::mutex mu;
  static bool done[64][2][2];
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int hi = head_dim == 128 ? 1 : 0, ni = nsess_template == 1 ? 0 : 1;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev][hi][ni]) return cudaSuccess;
  cudaError_t e = sr::attn_prepare(head_dim, nsess_template);
  if (e == cudaSuccess) done[dev][hi][ni] = true;
  return e;
}

// What one attention call of a session sees: the chunk's query/key rows and
// how many of the most recent committed frames are visible.
struct ChunkView {
  int64_t lq;         // chunk rows, frames * T
  int64_t hist;       // visible history: the last `hist` committed frames (host-state calls)
  bool dev = false;   // device-state call: the kernel derives the history from the frame counter
  int32_t hist_req = -1;   // ... of this many frames (-1: every occupied slot)
};

// The plain calls: the configured chunk length and every occupied slot.
ChunkView default_view(const sr_session* s) {
  return {s->lq, std::min<int64_t>(s->n_committed, s->cfg.window_frames)};
}

// Ring rows holding frames n-hist .. n-1, as one or two contiguous ranges
// [r0, r0 + c0) and [0, c1) (the second when they wrap around the end of the
// ring). All W slots at once are one range whatever the order.
void ring_ranges(const sr_session* s, int64_t hist, int64_t& r0, int64_t& c0, int64_t& c1) {
  const int64_t W = s->cfg.window_frames, T = s->tokens_per_frame;
  r0 = c0 = c1 = 0;
  if (hist <= 0 || W == 0) return;
  if (hist >= W) {
    c0 = W * T;
    return;
  }
  const int64_t start = (s->n_committed - hist) % W;
  if (start + hist <= W) {
    r0 = start * T;
    c0 = hist * T;
  } else {
    r0 = start * T;
    c0 = (W - start) * T;
    c1 = (start + hist - W) * T;
  }
}

// One key/value segment of a query group: rows [0, rows) of the buffers k, v.
struct Segment {
  const void* k;
  const void* v;
  int64_t rows;
};

// Encode a query group's four key/value segments (empty ones get no map),
// and its query rows [row0, row0 + lq) of the packed q / o.
sr_status encode_group(sr::AttnSession& out, const Segment (&seg)[sr::kSegs], int64_t row_elems, int64_t row0,
                       int64_t lq, sr_session* cache) {
  std::memset(&out, 0, sizeof(out));
  for (int i = 0; i < sr::kSegs; ++i) {
    out.seg_rows[i] = static_cast<int32_t>(seg[i].rows);
    if (seg[i].rows > 0 && (!encode_cached(cache, &out.kmap[i], seg[i].k, seg[i].rows, row_elems) ||
                            !encode_cached(cache, &out.vmap[i], seg[i].v, seg[i].rows, row_elems)))
      return SR_ERR_CUDA;
  }
  out.q_row0 = static_cast<int32_t>(row0);
  out.lq = static_cast<int32_t>(lq);
  out.nqb = static_cast<int32_t>((lq + 255) / 256);
  const int64_t rem = lq % 256;
  out.ntail = (rem > 0 && rem <= 128) ? 1 : 0;   // a single-tile last block
  out.nfull = out.nqb - out.ntail;
  return SR_OK;
}

// Place a query group's units: its whole blocks after `full` units, its
// single-tile last blocks after `tails` last-block units (both advance).
void place_units(sr::AttnSession& g, int n_heads, int& full, int& tails) {
  g.unit_begin = full;
  g.tail_begin = tails;
  full += n_heads * g.nfull;
  tails += n_heads * g.ntail;
}

// The packed unit ranges of the launch's query groups (after place_units).
template <int N>
void index_units(sr::AttnParams<N>& p) {
  for (int i = 0; i < p.n_sess; ++i) {
    p.whole_end[i] = p.sess[i].unit_begin + p.n_heads * p.sess[i].nfull;
    p.tail_end[i] = p.sess[i].tail_begin + p.n_heads * p.sess[i].ntail;
  }
}

// The launch's unit count, and the unit counter of a persistent launch: it
// lives at the start of the first group's workspace (none: one unit per CTA).
template <int N>
void set_units(sr::AttnParams<N>& p, int n_units, const sr_session* first) {
  index_units(p);
  p.n_units = n_units;
  if (first->buf.workspace != nullptr && p.sess[0].ws_ctr != nullptr) {
    p.unit_ctr = static_cast<unsigned long long*>(first->buf.workspace);
    p.epoch = p.sess[0].epoch;
  } else {
    p.unit_ctr = nullptr;
    p.epoch = 0;
  }
}

const char* bank_ptr(const void* bank, const sr_session* s, int step) {
  const size_t row_bytes = static_cast<size_t>(s->cfg.n_heads) * s->cfg.head_dim * 2;
  return static_cast<const char*>(bank) + static_cast<size_t>(step) * s->cfg.n_sink * row_bytes;
}

// A new epoch for this call's counters (27 bits: the key-split counter keeps
// its arrivals in the low 4 bits of an int32; never 0, the cleared value).
// The counters are raised to a call's epoch with atomicMax, so a count left by
// a call that stopped early (a device timeout) under a high epoch would outlast
// the wrap back to 1: after a wrap the counters are cleared on the stream
// before the next launch (clear_stale_counters).
int32_t next_epoch(sr_session* s) {
  s->epoch = (s->epoch + 1) & 0x07FFFFFF;
  if (s->epoch == 0) {
    s->epoch = 1;
    s->counters_stale = true;
  }
  return s->epoch;
}

// Zero the launch-wide unit counter and the per-head arrival counters of a
// session's workspace if its epoch wrapped since the last launch.
sr_status clear_stale_counters(sr_session* s, cudaStream_t st) {
  if (!s->counters_stale) return SR_OK;
  if (s->buf.workspace != nullptr &&
      sr::launch_zero_words(static_cast<int32_t*>(s->buf.workspace),
                            static_cast<int>(sr::kWsUnitCtrBytes / 4) + s->cfg.n_heads, st) != cudaSuccess)
    return SR_ERR_CUDA;
  s->counters_stale = false;
  return SR_OK;
}

// Fill one session's segment maps for `step` (rows of the chunk taken from
// k, v at row offset `row0` of a packed tensor).
sr_status fill_session(sr::AttnSession& out, sr_session* s, const ChunkView& view, int step, const void* k,
                       const void* v, int64_t row0) {
  const int64_t row_elems = static_cast<int64_t>(s->cfg.n_heads) * s->cfg.head_dim;
  const size_t row_bytes = static_cast<size_t>(row_elems) * 2;
  int64_t r0 = 0, c0 = 0, c1 = 0;
  if (view.dev) {
    // both ring segments map the whole ring; the kernel picks the rows
    c0 = c1 = s->cfg.window_frames * s->tokens_per_frame;
  } else {
    ring_ranges(s, view.hist, r0, c0, c1);
  }
  const size_t ring_off = static_cast<size_t>(r0) * row_bytes;
  const Segment seg[sr::kSegs] = {
      {bank_ptr(s->buf.sink_k, s, step), bank_ptr(s->buf.sink_v, s, step), s->cfg.n_sink},
      {static_cast<const char*>(s->buf.ring_k) + ring_off, static_cast<const char*>(s->buf.ring_v) + ring_off, c0},
      {s->buf.ring_k, s->buf.ring_v, c1},
      {static_cast<const char*>(k) + static_cast<size_t>(row0) * row_bytes,
       static_cast<const char*>(v) + static_cast<size_t>(row0) * row_bytes, view.lq}};
  sr_status st = encode_group(out, seg, row_elems, row0, view.lq, s);
  if (st != SR_OK) return st;
  if (view.dev) {
    out.dev_n = s->buf.frame_counter;
    out.hist_req = view.hist_req;
    out.ring_W = s->cfg.window_frames;
    out.ring_T = static_cast<int32_t>(s->tokens_per_frame);
  }
  if (s->buf.workspace) {
    char* ws = static_cast<char*>(s->buf.workspace);
    out.ws_ctr = reinterpret_cast<int32_t*>(ws + sr::kWsUnitCtrBytes);
    out.ws_part = reinterpret_cast<float*>(ws + sr::ws_counter_bytes(s->cfg.n_heads));
    out.epoch = next_epoch(s);
  }
  return SR_OK;
}

// Key tiles a session's chunk attends over (sink bank + visible ring + chunk).
int64_t key_tiles(const sr_session* s, const ChunkView& view) {
  int64_t r0 = 0, c0 = 0, c1 = 0;
  // a device-state call may see anything from no ring frame up: plan for none
  if (!view.dev) ring_ranges(s, view.hist, r0, c0, c1);
  const int64_t rows[4] = {s->cfg.n_sink, c0, c1, view.lq};
  int64_t n = 0;
  for (int64_t r : rows) n += (r + 127) / 128;
  return n;
}

// Longest-first dispatch of units with the given costs (in key-tile
// iterations of a whole block) to whichever of G SMs frees up first; the
// makespan.
double dispatch_makespan(const std::vector<double>& costs, int G) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int g = 0; g < G; ++g) free_at.push(0.0);
  for (double c : costs) {
    const double t0 = free_at.top();
    free_at.pop();
    free_at.push(t0 + c);
  }
  double t = 0;
  while (!free_at.empty()) {
    t = std::max(t, free_at.top());
    free_at.pop();
  }
  return t;
}

// Whole blocks left over in a last wave that is at most half full (0 when
// the blocks do not fill one wave, or fill the last one more than half): the
// candidates for running as single-tile units. A launch smaller than a wave
// shares the GPU with the previous and next launches of the stream, which the
// simulation does not see, and a fuller last wave is better left whole
// (measured on the decoder's shifted layers: converting them made a layer up
// to 15 % slower).
int64_t sparse_last_wave(int64_t whole, int G) {
  if (whole < G) return 0;
  const int64_t left = whole % G;
  return left <= G / 2 ? left : 0;
}

// Costs measured on GB300, in iterations of a whole block: a whole block
// walks all its key tiles; a single-tile unit walks half of them in split
// mode at 1.33x the cost per tile, plus about half an iteration of set-up;
// a key-range part of a last block walks its share the same way, plus half
// an iteration of merge when the block is split.
double single_tile_cost(double tiles) { return std::ceil(tiles / 2.0) * 1.33 + 0.5; }
double part_cost(double tiles, int k) {
  return std::ceil(std::ceil(tiles / k) / 2.0) * 1.33 + 0.5 + (k > 1 ? 0.5 : 0.0);
}

// The launch plan of a batch of query groups (in unit order): key-range parts
// per single-tile last block (k; only when every group ends in a single tile
// and has a workspace: in a batch that mixes them, such as the decoder's edge
// windows, parts of the few short last blocks cost more in set-up than they
// save) and how many of the last whole blocks run as two single-tile units
// each (c; when the whole blocks leave a partly filled last wave, those few
// blocks would otherwise run alone while the other SMs idle). The dispatch
// simulation decides; more parts must shorten the makespan by 0.5 %, a
// conversion by 2 %.
void choose_batch_plan(sr_session* const* ss, const ChunkView* views, const int* order, int n, int& k_out,
                       int& c_out) {
  const int G = sr::sm_count();
  const int forced = ss[order[0]]->cfg.tail_split;
  std::vector<double> whole, tails;   // whole-block costs in unit order; tiles of each single-tile last block
  bool all_single = true;
  int64_t min_kv = INT64_MAX;
  for (int r = 0; r < n; ++r) {
    const sr_session* s = ss[order[r]];
    const ChunkView& view = views[order[r]];
    const int64_t rem = view.lq % 256;
    const bool single = rem > 0 && rem <= 128;
    const double tiles = static_cast<double>(key_tiles(s, view));
    const int64_t blocks = static_cast<int64_t>(s->cfg.n_heads) * ((view.lq + 255) / 256 - (single ? 1 : 0));
    whole.insert(whole.end(), static_cast<size_t>(blocks), tiles);
    if (single) {
      tails.insert(tails.end(), static_cast<size_t>(s->cfg.n_heads), tiles);
      min_kv = std::min(min_kv, key_tiles(s, view));
    }
    if (!single || !s->buf.workspace) all_single = false;
  }
  int k_lo = 1, k_hi = 1;
  if (all_single && !tails.empty()) {
    const int cap = static_cast<int>(std::min<int64_t>(SR_MAX_TAIL_SPLIT, min_kv));
    k_lo = forced > 0 ? std::max(1, std::min(forced, cap)) : 1;
    k_hi = forced > 0 ? k_lo : cap;
  }
  const int64_t left = sparse_last_wave(static_cast<int64_t>(whole.size()), G);
  int best_k = k_lo, best_c = 0;
  double best_t = 0;
  bool have = false;
  std::vector<double> units;
  for (int64_t c : {int64_t(0), left}) {
    if (have && c == 0) break;   // left == 0: nothing to convert
    for (int k = k_lo; k <= k_hi; ++k) {
      units.clear();
      const size_t keep = whole.size() - static_cast<size_t>(c);
      units.insert(units.end(), whole.begin(), whole.begin() + static_cast<std::ptrdiff_t>(keep));
      for (size_t i = keep; i < whole.size(); ++i) units.insert(units.end(), 2, single_tile_cost(whole[i]));
      for (double t : tails) units.insert(units.end(), static_cast<size_t>(k), part_cost(t, k));
      const double t = dispatch_makespan(units, G);
      const bool better = !have || (c == best_c ? t < best_t * 0.995 : t < best_t * 0.98);
      if (better) {
        best_t = t;
        best_k = k;
        best_c = static_cast<int>(c);
        have = true;
      }
    }
  }
  k_out = best_k;
  c_out = best_c;
}

// The plan of one query group, from the launch's numbers alone: the same
// choice as choose_batch_plan for a batch of one.
void plan_units(int H, int64_t lq, int64_t tiles, bool has_ws, int forced, int G, int& k_out, int& c_out) {
  const int64_t rem = lq % 256;
  const bool single = rem > 0 && rem <= 128;
  const int64_t whole = static_cast<int64_t>(H) * ((lq + 255) / 256 - (single ? 1 : 0));
  int k_lo = 1, k_hi = 1;
  if (single && has_ws) {
    const int cap = static_cast<int>(std::min<int64_t>(SR_MAX_TAIL_SPLIT, tiles));
    k_lo = forced > 0 ? std::max(1, std::min(forced, cap)) : 1;
    k_hi = forced > 0 ? k_lo : cap;
  }
  const int64_t left = sparse_last_wave(whole, G);
  const double t_full = static_cast<double>(tiles);
  int best_k = k_lo, best_c = 0;
  double best_t = 0;
  bool have = false;
  std::vector<double> units;
  for (int64_t c : {int64_t(0), left}) {
    if (have && c == 0) break;   // left == 0: nothing to convert
    for (int k = k_lo; k <= k_hi; ++k) {
      units.assign(static_cast<size_t>(whole - c), t_full);
      units.insert(units.end(), static_cast<size_t>(2 * c), single_tile_cost(t_full));
      if (single) units.insert(units.end(), static_cast<size_t>(H) * k, part_cost(t_full, k));
      const double t = dispatch_makespan(units, G);
      // more parts or a conversion must gain clearly: each part and unit costs set-up
      const bool better = !have || (c == best_c ? t < best_t * 0.995 : t < best_t * 0.98);
      if (better) {
        best_t = t;
        best_k = k;
        best_c = static_cast<int>(c);
        have = true;
      }
    }
  }
  k_out = best_k;
  c_out = best_c;
}

// The plan of a one-group launch, kept per session for the shape it was
// made for (the simulation runs once per shape, not once per call).
void choose_plan(sr_session* s, const ChunkView& view, int& k_out, int& c_out) {
  const int G = sr::sm_count();
  const int64_t tiles = key_tiles(s, view);
  const int64_t key[4] = {view.lq, tiles, G, s->buf.workspace != nullptr};
  if (!std::equal(key, key + 4, s->plan_key)) {
    plan_units(s->cfg.n_heads, view.lq, tiles, s->buf.workspace != nullptr, s->cfg.tail_split, G, s->plan_split,
               s->plan_conv);
    std::copy(key, key + 4, s->plan_key);
  }
  k_out = s->plan_split;
  c_out = s->plan_conv;
}

}  // namespace

namespace sr {

int sm_count() {
  static int counts[64];
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return 152;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    counts[dev] = n;
  }
  return counts[dev];
}

int session_heads(const sr_session* s) { return s->cfg.n_heads; }

sr_status attention_scratch_check(const sr_session* s, int32_t step, const void* q, const void* k, const void* v,
                                  const void* o, const float* lse, uint64_t scratch_bytes) {
  if (!s || !q || !k || !v || !o) return SR_ERR_INVALID_ARG;
  if (step < 0 || step >= s->cfg.n_steps) return SR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return SR_ERR_ALIGN;
  uint64_t need = 0;
  if (sr_workspace_bytes(&s->cfg, &need) != SR_OK || need > scratch_bytes) return SR_ERR_UNSUPPORTED;
  return SR_OK;
}

sr_status attention_into_scratch(sr_session* s, int32_t step, const void* q, const void* k, const void* v, void* o,
                                 float* lse, void* stream, void* scratch) {
  if (ensure_attn_attr(s->cfg.head_dim, 1) != cudaSuccess) return SR_ERR_CUDA;
  AttnParams<1> p;                                  // on the stack: nothing is allocated
  std::memset(&p, 0, sizeof(p));
  const int64_t row_elems = static_cast<int64_t>(s->cfg.n_heads) * s->cfg.head_dim;
  if (!encode_cached(s, &p.qmap, q, s->lq, row_elems))
    return SR_ERR_CUDA;
  // the scratch stands in for the session's workspace for this call only
  void* own = s->buf.workspace;
  s->buf.workspace = scratch;
  const ChunkView view = default_view(s);
  sr_status st = fill_session(p.sess[0], s, view, step, k, v, 0);
  int split = 1, conv = 0;
  if (st == SR_OK) choose_plan(s, view, split, conv);
  s->buf.workspace = own;
  if (st != SR_OK) return st;
  int full = 0, tails = 0;
  place_units(p.sess[0], s->cfg.n_heads, full, tails);
  p.n_full_units = full;
  p.n_conv = conv;
  p.tail_split = split;
  const int n_units = full + conv + tails * split;
  p.n_sess = 1;
  p.n_heads = s->cfg.n_heads;
  p.scale_log2 = s->scale * 1.4426950408889634f;
  p.lse_ld = lse ? static_cast<int32_t>(s->lq) : 0;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err_word = s->buf.err_word;
  p.timeout_ns = s->cfg.wait_timeout_ns;
  s->buf.workspace = scratch;
  set_units(p, n_units, s);
  s->buf.workspace = own;
  return launch_attention_1(p, s->cfg.head_dim, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SR_OK
                                                                                                  : SR_ERR_CUDA;
}

}  // namespace sr

extern "C" {

const char* sr_status_string(sr_status st) {
  switch (st) {
    case SR_OK: return "ok";
    case SR_ERR_INVALID_ARG: return "invalid argument";
    case SR_ERR_UNSUPPORTED: return "unsupported configuration";
    case SR_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case SR_ERR_STATE: return "call not allowed in the session's state";
    case SR_ERR_CUDA: return "CUDA call or kernel launch failed";
    case SR_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

sr_status sr_device_error_status(int32_t v) { return v == SR_DEVERR_NONE ? SR_OK : SR_ERR_TIMEOUT; }

sr_status sr_plan_attention(int32_t n_heads, int64_t lq, int64_t key_tiles, int32_t has_workspace,
                            int32_t tail_split, int32_t sm_count, int32_t* parts, int32_t* whole_as_tiles,
                            int64_t* n_units) {
  if (!parts || !whole_as_tiles || !n_units || n_heads < 1 || lq < 1 || key_tiles < 1 || tail_split < 0 ||
      tail_split > SR_MAX_TAIL_SPLIT || lq > (int64_t(1) << 28) || key_tiles > (int64_t(1) << 24))
    return SR_ERR_INVALID_ARG;
  const int G = sm_count > 0 ? sm_count : sr::sm_count();
  int k = 1, c = 0;
  plan_units(n_heads, lq, key_tiles, has_workspace != 0, tail_split, G, k, c);
  const int64_t rem = lq % 256;
  const bool single = rem > 0 && rem <= 128;
  const int64_t whole = static_cast<int64_t>(n_heads) * ((lq + 255) / 256 - (single ? 1 : 0));
  *parts = k;
  *whole_as_tiles = c;
  *n_units = whole + c + (single ? static_cast<int64_t>(n_heads) * k : 0);
  return SR_OK;
}

sr_status sr_workspace_bytes(const sr_config* cfg, uint64_t* bytes) {
  if (!cfg || !bytes) return SR_ERR_INVALID_ARG;
  sr_status st = validate_config(*cfg);
  if (st != SR_OK) return st;
  *bytes = sr::ws_counter_bytes(cfg->n_heads) +
           static_cast<uint64_t>(cfg->n_heads) * sr::ws_partial_floats_per_head(cfg->head_dim) * sizeof(float);
  return SR_OK;
}

sr_status sr_session_init(const sr_config* cfg, const sr_buffers* bufs, const void* sink_k_src,
                          const void* sink_v_src, void* stream, sr_session** out) {
  if (out) *out = nullptr;
  if (!cfg || !bufs || !out) return SR_ERR_INVALID_ARG;
  sr_status st = validate_config(*cfg);
  if (st != SR_OK) return st;
  const bool has_sink = cfg->n_sink > 0;
  const bool has_ring = cfg->window_frames > 0;
  if ((has_sink && (!bufs->sink_k || !bufs->sink_v)) || (has_ring && (!bufs->ring_k || !bufs->ring_v)) ||
      (has_ring && !bufs->slot_frame) || !bufs->err_word)
    return SR_ERR_INVALID_ARG;
  if ((sink_k_src == nullptr) != (sink_v_src == nullptr)) return SR_ERR_INVALID_ARG;
  if ((has_sink && (!aligned16(bufs->sink_k) || !aligned16(bufs->sink_v))) ||
      (has_ring && (!aligned16(bufs->ring_k) || !aligned16(bufs->ring_v))) ||
      (sink_k_src && (!aligned16(sink_k_src) || !aligned16(sink_v_src))) ||
      (reinterpret_cast<uintptr_t>(bufs->err_word) & 3u) ||
      (reinterpret_cast<uintptr_t>(bufs->workspace) & 255u) ||
      (reinterpret_cast<uintptr_t>(bufs->slot_frame) & 3u) ||
      (reinterpret_cast<uintptr_t>(bufs->frame_counter) & 7u))
    return SR_ERR_ALIGN;

  sr_session* s = new (std::nothrow) sr_session;
  if (!s) return SR_ERR_INVALID_ARG;
  std::memset(s, 0, sizeof(*s));
  s->cfg = *cfg;
  if (s->cfg.wait_timeout_ns == 0) s->cfg.wait_timeout_ns = kDefaultTimeoutNs;
  s->buf = *bufs;
  s->tokens_per_frame = static_cast<int64_t>(cfg->grid_h) * cfg->grid_w;
  s->lq = s->tokens_per_frame * cfg->chunk_frames;
  s->scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0f / std::sqrt(static_cast<float>(cfg->head_dim));
  s->n_committed = 0;
  sr::rope_phase_table(cfg->rope_base, cfg->head_dim, &s->phase);

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (sink_k_src && has_sink) {
    const size_t bytes = static_cast<size_t>(cfg->n_steps) * cfg->n_sink * cfg->n_heads * cfg->head_dim * 2;
    e = sr::launch_copy16(bufs->sink_k, sink_k_src, bytes, cs);
    if (e == cudaSuccess) e = sr::launch_copy16(bufs->sink_v, sink_v_src, bytes, cs);
  }
  if (e == cudaSuccess)
    e = sr::launch_init_ring_state(bufs->slot_frame, cfg->window_frames, bufs->err_word,
                                   static_cast<int32_t*>(bufs->workspace),
                                   static_cast<int>(sr::kWsUnitCtrBytes / 4) + cfg->n_heads, cs);
  if (e == cudaSuccess && bufs->frame_counter) {
    // device-state calls: the counter starts at 0, and ring tiles that straddle
    // the visible rows read zeros rather than whatever the buffers held
    e = cudaMemsetAsync(bufs->frame_counter, 0, sizeof(int64_t), cs);
    const size_t ring_bytes = static_cast<size_t>(cfg->window_frames) * s->tokens_per_frame * cfg->n_heads *
                              cfg->head_dim * 2;
    if (e == cudaSuccess && ring_bytes) e = cudaMemsetAsync(bufs->ring_k, 0, ring_bytes, cs);
    if (e == cudaSuccess && ring_bytes) e = cudaMemsetAsync(bufs->ring_v, 0, ring_bytes, cs);
  }
  if (e == cudaSuccess) e = ensure_attn_attr(cfg->head_dim, 1);
  if (e == cudaSuccess) e = ensure_attn_attr(cfg->head_dim, sr::kAttnMaxBatch);
  if (e != cudaSuccess) {
    delete s;
    return SR_ERR_CUDA;
  }
  *out = s;
  return SR_OK;
}

sr_status sr_session_restore(sr_session* s, int64_t n_committed) {
  if (!s || n_committed < 0 || n_committed > kMaxFrames) return SR_ERR_INVALID_ARG;
  s->n_committed = n_committed;
  return SR_OK;
}

sr_status sr_session_frames(const sr_session* s, int64_t* n) {
  if (!s || !n) return SR_ERR_INVALID_ARG;
  *n = s->n_committed;
  return SR_OK;
}

// Frames a single call may carry: the limits sr_session_init applies to the
// configured chunk length.
static bool frames_ok(const sr_session* s, int64_t n_frames) {
  const int64_t row = static_cast<int64_t>(s->cfg.n_heads) * s->cfg.head_dim;
  const int64_t limit = int64_t(1) << 30;
  if (n_frames < 1 || n_frames > limit) return false;
  const int64_t lq = n_frames * s->tokens_per_frame;
  return lq <= limit / 4 && lq * row <= limit;
}

// RoPE (mode 0) or commit (mode 1) of `n_frames` frames; frame f is the
// stream's frame first_frame + f, with time t_clock0 + first_frame + f (the
// chunk calls pass n_committed).
static sr_status rope_common(sr_session* s, int64_t first_frame, int64_t n_frames, const void* a_src,
                             const void* b_src, void* a_dst, void* b_dst, int mode, void* stream,
                             const int64_t* dev_n = nullptr) {
  sr::RopeParams p;
  std::memset(&p, 0, sizeof(p));
  int64_t first = 0;   // first frame of the chunk that is processed
  if (mode == 1 && n_frames > s->cfg.window_frames) first = n_frames - s->cfg.window_frames;
  const size_t skip = static_cast<size_t>(first * s->tokens_per_frame) * s->cfg.n_heads * s->cfg.head_dim;
  p.src0 = static_cast<const __nv_bfloat16*>(a_src) + skip;
  p.src1 = static_cast<const __nv_bfloat16*>(b_src) + skip;
  p.dst0 = static_cast<__nv_bfloat16*>(a_dst);
  p.dst1 = static_cast<__nv_bfloat16*>(b_dst);
  p.slot_frame = s->buf.slot_frame;
  p.n_committed = first_frame + first;
  p.n_tok = static_cast<int32_t>((n_frames - first) * s->tokens_per_frame);
  p.n_heads = s->cfg.n_heads;
  p.tokens_per_frame = static_cast<int32_t>(s->tokens_per_frame);
  p.grid_w = s->cfg.grid_w;
  p.window_frames = s->cfg.window_frames;
  p.chunk_frames = static_cast<int32_t>(n_frames - first);
  p.t_clock0 = s->cfg.t_clock0;
  p.mode = mode;
  p.phase = s->phase;
  p.dev_n = dev_n;   // when set, first_frame is an offset from the device counter
  cudaError_t e = sr::launch_rope(p, s->cfg.head_dim, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SR_OK : SR_ERR_CUDA;
}

sr_status sr_rope3d_qk_frames(sr_session* s, int32_t n_frames, void* q, void* k, void* stream) {
  if (!s || !frames_ok(s, n_frames)) return SR_ERR_INVALID_ARG;
  if ((q && !aligned16(q)) || (k && !aligned16(k))) return SR_ERR_ALIGN;
  if (!q && !k) return SR_OK;
  if (q && k) return rope_common(s, s->n_committed, n_frames, q, k, q, k, 0, stream);
  // One tensor: pass it as both operands. Each 16-byte vector is loaded by one
  // thread into two registers before either store, so both stores write the
  // same once-rotated value.
  void* x = q ? q : k;
  return rope_common(s, s->n_committed, n_frames, x, x, x, x, 0, stream);
}

sr_status sr_rope3d_qk_at(sr_session* s, int64_t first_frame, int32_t n_frames, void* q, void* k, void* stream) {
  if (!s || !frames_ok(s, n_frames)) return SR_ERR_INVALID_ARG;
  if (first_frame < -(int64_t(1) << 40) || first_frame > (int64_t(1) << 40)) return SR_ERR_INVALID_ARG;
  if ((q && !aligned16(q)) || (k && !aligned16(k))) return SR_ERR_ALIGN;
  if (!q && !k) return SR_OK;
  if (q && k) return rope_common(s, first_frame, n_frames, q, k, q, k, 0, stream);
  void* x = q ? q : k;
  return rope_common(s, first_frame, n_frames, x, x, x, x, 0, stream);
}

sr_status sr_rope3d_qk(sr_session* s, void* q, void* k, void* stream) {
  if (!s) return SR_ERR_INVALID_ARG;
  return sr_rope3d_qk_frames(s, s->cfg.chunk_frames, q, k, stream);
}

sr_status sr_cache_commit_frames(sr_session* s, int32_t n_frames, const void* k_raw, const void* v, void* stream) {
  if (!s || !k_raw || !v || !frames_ok(s, n_frames)) return SR_ERR_INVALID_ARG;
  if (!aligned16(k_raw) || !aligned16(v)) return SR_ERR_ALIGN;
  if (s->n_committed + n_frames > kMaxFrames) return SR_ERR_STATE;
  if (s->cfg.window_frames == 0) {
    s->n_committed += n_frames;
    return SR_OK;
  }
  sr_status st = rope_common(s, s->n_committed, n_frames, k_raw, v, s->buf.ring_k, s->buf.ring_v, 1, stream);
  if (st == SR_OK) s->n_committed += n_frames;
  return st;
}

sr_status sr_cache_commit(sr_session* s, const void* k_raw, const void* v, void* stream) {
  if (!s) return SR_ERR_INVALID_ARG;
  return sr_cache_commit_frames(s, s->cfg.chunk_frames, k_raw, v, stream);
}

static sr_status attention_view(sr_session* s, const ChunkView& view, int32_t step, const void* q, const void* k,
                                const void* v, void* o, float* lse, void* stream) {
  if (!s || !q || !k || !v || !o) return SR_ERR_INVALID_ARG;
  if (step < 0 || step >= s->cfg.n_steps) return SR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return SR_ERR_ALIGN;
  if (ensure_attn_attr(s->cfg.head_dim, 1) != cudaSuccess) return SR_ERR_CUDA;
  auto* p = new (std::nothrow) sr::AttnParams<1>;
  if (!p) return SR_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  const int64_t row_elems = static_cast<int64_t>(s->cfg.n_heads) * s->cfg.head_dim;
  sr_status st = SR_OK;
  if (!encode_cached(s, &p->qmap, q, view.lq, row_elems))
    st = SR_ERR_CUDA;
  if (st == SR_OK) st = fill_session(p->sess[0], s, view, step, k, v, 0);
  int n_units = 0;
  if (st == SR_OK) {
    // whole 256-row blocks first (longest units), then single-tile last blocks
    int full = 0, tails = 0;
    place_units(p->sess[0], s->cfg.n_heads, full, tails);
    p->n_full_units = full;
    int split = 1, conv = 0;
    choose_plan(s, view, split, conv);
    p->n_conv = conv;
    p->tail_split = split;
    n_units = full + conv + tails * split;
    p->n_sess = 1;
    p->n_heads = s->cfg.n_heads;
    p->scale_log2 = s->scale * 1.4426950408889634f;
    p->lse_ld = lse ? static_cast<int32_t>(view.lq) : 0;
    p->o = static_cast<__nv_bfloat16*>(o);
    p->lse = lse;
    p->err_word = s->buf.err_word;
    p->timeout_ns = s->cfg.wait_timeout_ns;
    set_units(*p, n_units, s);
    st = clear_stale_counters(s, static_cast<cudaStream_t>(stream));
    if (st == SR_OK &&
        sr::launch_attention_1(*p, s->cfg.head_dim, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      st = SR_ERR_CUDA;
  }
  delete p;
  return st;
}

sr_status sr_chunk_attention(sr_session* s, int32_t step, const void* q, const void* k, const void* v, void* o,
                             float* lse, void* stream) {
  if (!s) return SR_ERR_INVALID_ARG;
  return attention_view(s, default_view(s), step, q, k, v, o, lse, stream);
}

sr_status sr_chunk_attention_frames(sr_session* s, int32_t step, int32_t n_frames, int32_t hist_frames,
                                    const void* q, const void* k, const void* v, void* o, float* lse,
                                    void* stream) {
  if (!s || !frames_ok(s, n_frames)) return SR_ERR_INVALID_ARG;
  const int64_t occupied = std::min<int64_t>(s->n_committed, s->cfg.window_frames);
  if (hist_frames < -1 || hist_frames > occupied) return SR_ERR_INVALID_ARG;
  const ChunkView view{n_frames * s->tokens_per_frame, hist_frames == -1 ? occupied : hist_frames};
  return attention_view(s, view, step, q, k, v, o, lse, stream);
}

sr_status sr_rope3d_qk_dev(sr_session* s, int32_t n_frames, void* q, void* k, void* stream) {
  if (!s || !frames_ok(s, n_frames)) return SR_ERR_INVALID_ARG;
  if (!s->buf.frame_counter) return SR_ERR_STATE;
  if ((q && !aligned16(q)) || (k && !aligned16(k))) return SR_ERR_ALIGN;
  if (!q && !k) return SR_OK;
  if (q && k) return rope_common(s, 0, n_frames, q, k, q, k, 0, stream, s->buf.frame_counter);
  void* x = q ? q : k;
  return rope_common(s, 0, n_frames, x, x, x, x, 0, stream, s->buf.frame_counter);
}

sr_status sr_chunk_attention_dev(sr_session* s, int32_t step, int32_t n_frames, int32_t hist_frames,
                                 const void* q, const void* k, const void* v, void* o, float* lse, void* stream) {
  if (!s || !frames_ok(s, n_frames)) return SR_ERR_INVALID_ARG;
  if (!s->buf.frame_counter) return SR_ERR_STATE;
  if (hist_frames < -1 || hist_frames > s->cfg.window_frames) return SR_ERR_INVALID_ARG;
  ChunkView view{n_frames * s->tokens_per_frame, 0};
  view.dev = true;
  view.hist_req = hist_frames;
  return attention_view(s, view, step, q, k, v, o, lse, stream);
}

sr_status sr_cache_commit_dev(sr_session* s, int32_t n_frames, const void* k_raw, const void* v, void* stream) {
  if (!s || !k_raw || !v || !frames_ok(s, n_frames)) return SR_ERR_INVALID_ARG;
  if (!s->buf.frame_counter) return SR_ERR_STATE;
  if (!aligned16(k_raw) || !aligned16(v)) return SR_ERR_ALIGN;
  if (s->n_committed + n_frames > kMaxFrames) return SR_ERR_STATE;
  sr_status st = SR_OK;
  if (s->cfg.window_frames > 0)   // frame times and slots from the device counter (offset 0)
    st = rope_common(s, 0, n_frames, k_raw, v, s->buf.ring_k, s->buf.ring_v, 1, stream, s->buf.frame_counter);
  if (st == SR_OK &&
      sr::launch_advance_frames(s->buf.frame_counter, n_frames, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    st = SR_ERR_CUDA;
  if (st == SR_OK) s->n_committed += n_frames;   // the host mirror follows eager calls, not graph replays
  return st;
}

sr_status sr_window_attention(sr_session* s, int32_t step, int32_t moving_frames, int32_t with_prefix,
                              const void* q, const void* k_moving, const void* v_moving, void* o, float* lse,
                              void* stream) {
  if (!s || !q || !k_moving || !v_moving || !o || !frames_ok(s, moving_frames)) return SR_ERR_INVALID_ARG;
  if (step < 0 || step >= s->cfg.n_steps) return SR_ERR_INVALID_ARG;
  if (with_prefix && s->cfg.n_sink == 0) return SR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_moving) || !aligned16(v_moving) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return SR_ERR_ALIGN;
  const int64_t P = with_prefix ? s->cfg.n_sink : 0;
  const int64_t M = static_cast<int64_t>(moving_frames) * s->tokens_per_frame;
  const int64_t row_elems = static_cast<int64_t>(s->cfg.n_heads) * s->cfg.head_dim;
  if ((P + M) * row_elems > (int64_t(1) << 31) || P + M > (int64_t(1) << 28)) return SR_ERR_INVALID_ARG;
  if (ensure_attn_attr(s->cfg.head_dim, sr::kAttnMaxBatch) != cudaSuccess) return SR_ERR_CUDA;
  auto* p = new (std::nothrow) sr::AttnParams<sr::kAttnMaxBatch>;
  if (!p) return SR_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  sr_status st = SR_OK;
  if (!encode_cached(s, &p->qmap, q, P + M, row_elems))
    st = SR_ERR_CUDA;
  // Two query groups in one launch. Moving rows (longest key range first):
  // the bank of the step and the moving rows themselves. Prefix rows: the
  // bank alone -- the asymmetric mask as a choice of key set.
  const char* bk = bank_ptr(s->buf.sink_k, s, step);
  const char* bv = bank_ptr(s->buf.sink_v, s, step);
  const Segment moving[sr::kSegs] = {{bk, bv, s->cfg.n_sink}, {nullptr, nullptr, 0}, {nullptr, nullptr, 0},
                                     {k_moving, v_moving, M}};
  const Segment prefix[sr::kSegs] = {{bk, bv, s->cfg.n_sink}, {nullptr, nullptr, 0}, {nullptr, nullptr, 0},
                                     {nullptr, nullptr, 0}};
  int n = 0, full = 0, tails = 0;
  if (st == SR_OK) st = encode_group(p->sess[n++], moving, row_elems, P, M, s);
  if (st == SR_OK && P > 0) st = encode_group(p->sess[n++], prefix, row_elems, 0, P, s);
  if (st == SR_OK) {
    for (int i = 0; i < n; ++i) place_units(p->sess[i], s->cfg.n_heads, full, tails);
    p->n_full_units = full;
    p->tail_split = 1;   // the groups share one session: no key-split workspace
    p->n_sess = n;
    p->n_heads = s->cfg.n_heads;
    p->scale_log2 = s->scale * 1.4426950408889634f;
    p->lse_ld = lse ? static_cast<int32_t>(P + M) : 0;
    p->o = static_cast<__nv_bfloat16*>(o);
    p->lse = lse;
    p->err_word = s->buf.err_word;
    p->timeout_ns = s->cfg.wait_timeout_ns;
    // no key-range parts (the groups share one session); with a workspace the
    // launch is persistent, and a one-group launch may balance its last wave
    int conv = 0;
    if (n == 1) {
      int k = 1;
      const int64_t tiles = (s->cfg.n_sink + 127) / 128 + (M + 127) / 128;
      plan_units(s->cfg.n_heads, M, tiles, false, 0, sr::sm_count(), k, conv);
    }
    p->n_conv = conv;
    p->n_units = full + conv + tails;
    index_units(*p);
    if (s->buf.workspace) {
      p->unit_ctr = static_cast<unsigned long long*>(s->buf.workspace);
      p->epoch = next_epoch(s);
    }
    st = clear_stale_counters(s, static_cast<cudaStream_t>(stream));
    if (st == SR_OK &&
        sr::launch_attention_n(*p, s->cfg.head_dim, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      st = SR_ERR_CUDA;
  }
  delete p;
  return st;
}

sr_status sr_chunk_attention_batch(sr_session* const* sessions, int32_t n, int32_t step, const void* q,
                                   const void* k, const void* v, const int64_t* q_off, void* o, float* lse,
                                   void* stream) {
  if (!sessions || n < 1 || n > SR_MAX_BATCH || !q || !k || !v || !o || !q_off) return SR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return SR_ERR_ALIGN;
  const sr_session* s0 = sessions[0];
  if (!s0 || q_off[0] != 0) return SR_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const sr_session* s = sessions[i];
    if (!s || s->cfg.n_heads != s0->cfg.n_heads || s->cfg.head_dim != s0->cfg.head_dim || s->scale != s0->scale)
      return SR_ERR_INVALID_ARG;
    if (step < 0 || step >= s->cfg.n_steps) return SR_ERR_INVALID_ARG;
    if (q_off[i + 1] - q_off[i] != s->lq) return SR_ERR_INVALID_ARG;
  }
  const int64_t total = q_off[n];
  if (total > (int64_t(1) << 28)) return SR_ERR_INVALID_ARG;
  // longest key range first, so the biggest units start in the first wave
  int order[SR_MAX_BATCH];
  for (int i = 0; i < n; ++i) order[i] = i;
  auto lk = [&](int i) {
    const sr_session* s = sessions[i];
    return s->cfg.n_sink + std::min<int64_t>(s->n_committed, s->cfg.window_frames) * s->tokens_per_frame + s->lq;
  };
  std::stable_sort(order, order + n, [&](int a, int b) { return lk(a) > lk(b); });
  ChunkView views[SR_MAX_BATCH];
  for (int i = 0; i < n; ++i) views[i] = default_view(sessions[i]);

  if (ensure_attn_attr(s0->cfg.head_dim, sr::kAttnMaxBatch) != cudaSuccess) return SR_ERR_CUDA;
  auto* p = new (std::nothrow) sr::AttnParams<sr::kAttnMaxBatch>;
  if (!p) return SR_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  const int64_t row_elems = static_cast<int64_t>(s0->cfg.n_heads) * s0->cfg.head_dim;
  sr_status st = SR_OK;
  if (!encode_cached(sessions[order[0]], &p->qmap, q, total, row_elems))
    st = SR_ERR_CUDA;
  // units: every session's whole 256-row blocks (sessions by decreasing key
  // count), then the single-tile last blocks -- longest work first
  int full = 0, tails = 0;
  for (int r = 0; st == SR_OK && r < n; ++r) {
    const int i = order[r];
    st = fill_session(p->sess[r], sessions[i], views[i], step, k, v, q_off[i]);
    if (st == SR_OK) place_units(p->sess[r], s0->cfg.n_heads, full, tails);
  }
  int split = 1, conv = 0;
  if (st == SR_OK) choose_batch_plan(sessions, views, order, n, split, conv);
  const int units = full + conv + tails * split;
  if (st == SR_OK) {
    p->n_full_units = full;
    p->n_conv = conv;
    p->tail_split = split;
    p->n_sess = n;
    p->n_heads = s0->cfg.n_heads;
    p->scale_log2 = s0->scale * 1.4426950408889634f;
    p->lse_ld = lse ? static_cast<int32_t>(total) : 0;
    p->o = static_cast<__nv_bfloat16*>(o);
    p->lse = lse;
    p->err_word = s0->buf.err_word;
    p->timeout_ns = s0->cfg.wait_timeout_ns;
    set_units(*p, units, sessions[order[0]]);
    for (int i = 0; st == SR_OK && i < n; ++i) st = clear_stale_counters(sessions[i], static_cast<cudaStream_t>(stream));
    if (st == SR_OK &&
        sr::launch_attention_n(*p, s0->cfg.head_dim, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      st = SR_ERR_CUDA;
  }
  delete p;
  return st;
}

// A decoder layer's windows in one launch (sr_layer_rope_gather, mode 0, and
// sr_layer_commit, mode 1): validate that the sessions form one layer of the
// frame, then give each window a contiguous range of CTAs.
static sr_status layer_common(sr_session* const* ss, const sr_window* wins, int32_t n, int32_t fh, int32_t fw,
                              const void* s0, const void* s1, const void* s2, void* d0, void* d1, void* d2,
                              int mode, void* stream) {
  if (!ss || !wins || n < 1 || n > SR_MAX_LAYER_WINDOWS || fh < 1 || fw < 1 || !s0 || !s1) return SR_ERR_INVALID_ARG;
  if (mode == 0 && (!d0 || !d1 || ((s2 == nullptr) != (d2 == nullptr)))) return SR_ERR_INVALID_ARG;
  const void* ptrs[6] = {s0, s1, s2, d0, d1, d2};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return SR_ERR_ALIGN;
  const sr_session* a = ss[0];
  if (!a) return SR_ERR_INVALID_ARG;
  const int64_t F = a->cfg.chunk_frames;
  const int64_t row_elems = static_cast<int64_t>(a->cfg.n_heads) * a->cfg.head_dim;
  const int64_t frame_rows = static_cast<int64_t>(fh) * fw * F;
  if (frame_rows > (int64_t(1) << 28) || frame_rows * row_elems > (int64_t(1) << 40)) return SR_ERR_INVALID_ARG;
  int64_t packed = 0;
  for (int i = 0; i < n; ++i) {
    const sr_session* s = ss[i];
    const sr_window& w = wins[i];
    if (!s || s->cfg.n_heads != a->cfg.n_heads || s->cfg.head_dim != a->cfg.head_dim ||
        s->cfg.chunk_frames != F || s->cfg.t_clock0 != a->cfg.t_clock0 || s->cfg.rope_base != a->cfg.rope_base)
      return SR_ERR_INVALID_ARG;
    if (w.rows != s->cfg.grid_h || w.cols != s->cfg.grid_w || w.row0 < 0 || w.col0 < 0 ||
        static_cast<int64_t>(w.row0) + w.rows > fh || static_cast<int64_t>(w.col0) + w.cols > fw)
      return SR_ERR_INVALID_ARG;
    if (mode == 1 && s->n_committed + F > kMaxFrames) return SR_ERR_STATE;
    packed += s->lq;
  }
  if (packed > (int64_t(1) << 28)) return SR_ERR_INVALID_ARG;

  auto* p = new (std::nothrow) sr::LayerRopeParams;
  if (!p) return SR_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  p->phase = a->phase;
  p->src[0] = static_cast<const __nv_bfloat16*>(s0);
  p->src[1] = static_cast<const __nv_bfloat16*>(s1);
  p->src[2] = static_cast<const __nv_bfloat16*>(s2);
  p->dst[0] = static_cast<__nv_bfloat16*>(d0);
  p->dst[1] = static_cast<__nv_bfloat16*>(d1);
  p->dst[2] = static_cast<__nv_bfloat16*>(d2);
  p->frame_h = fh;
  p->frame_w = fw;
  p->n_heads = a->cfg.n_heads;
  p->t_clock0 = a->cfg.t_clock0;
  p->mode = mode;
  p->tokens_per_cta = sr::layer_tokens_per_cta(a->cfg.n_heads, a->cfg.head_dim, mode);
  int64_t ctas = 0, row = 0;
  int nw = 0;
  for (int i = 0; i < n; ++i) {
    const sr_session* s = ss[i];
    const int64_t W = s->cfg.window_frames;
    const int64_t first = (mode == 1 && F > W) ? F - W : 0;   // a commit keeps the chunk's last W frames
    const int64_t ntok = (mode == 1 && W == 0) ? 0 : (F - first) * s->tokens_per_frame;
    if (ntok > 0) {
      sr::LayerWindow& lw = p->win[nw++];
      lw.row0 = wins[i].row0;
      lw.col0 = wins[i].col0;
      lw.rows = wins[i].rows;
      lw.cols = wins[i].cols;
      lw.packed_row0 = row;
      lw.n_committed = s->n_committed;
      lw.ring_k = static_cast<__nv_bfloat16*>(s->buf.ring_k);
      lw.ring_v = static_cast<__nv_bfloat16*>(s->buf.ring_v);
      lw.slot_frame = s->buf.slot_frame;
      lw.window_frames = static_cast<int32_t>(W);
      lw.first_frame = static_cast<int32_t>(first);
      lw.cta_begin = static_cast<int32_t>(ctas);
      lw.n_tok = static_cast<int32_t>(ntok);
      ctas += (ntok + p->tokens_per_cta - 1) / p->tokens_per_cta;
    }
    row += s->lq;
  }
  p->n_windows = nw;
  sr_status st = SR_OK;
  if (ctas > (int64_t(1) << 30)) st = SR_ERR_INVALID_ARG;
  if (st == SR_OK && nw > 0 &&
      sr::launch_layer_rope(*p, a->cfg.head_dim, static_cast<int>(ctas), static_cast<cudaStream_t>(stream)) !=
          cudaSuccess)
    st = SR_ERR_CUDA;
  delete p;
  if (st == SR_OK && mode == 1)
    for (int i = 0; i < n; ++i) ss[i]->n_committed += F;
  return st;
}

sr_status sr_layer_rope_gather(sr_session* const* sessions, const sr_window* windows, int32_t n, int32_t frame_h,
                               int32_t frame_w, const void* q, const void* k, const void* v, void* q_packed,
                               void* k_packed, void* v_packed, void* stream) {
  return layer_common(sessions, windows, n, frame_h, frame_w, q, k, v, q_packed, k_packed, v_packed, 0, stream);
}

sr_status sr_layer_commit(sr_session* const* sessions, const sr_window* windows, int32_t n, int32_t frame_h,
                          int32_t frame_w, const void* k_raw, const void* v, void* stream) {
  return layer_common(sessions, windows, n, frame_h, frame_w, k_raw, v, nullptr, nullptr, nullptr, nullptr, 1,
                      stream);
}

// The unit rhythm of the teardown's shipped configuration: latents come in
// codec groups of five (the first covers one RGB frame, the others four);
// merging that one-frame latent into its neighbour makes units of 2, 1, 1, 1
// latents. Chunk 0 is the first window (bootstrap_units units, no history);
// chunk c >= 1 is chunk_units units and sees the window_units units before it.
static int64_t latents_before(int64_t u, bool merge) {   // latents in units 0 .. u-1
  if (!merge) return u;
  return u + (u + 3) / 4;   // units 0, 4, 8, ... below u hold one latent more
}

sr_status sr_plan_chunk(int32_t c, int32_t bootstrap_units, int32_t chunk_units, int32_t window_units,
                        int32_t sink_units, int32_t merge_single_frame_units, sr_chunk_plan* out) {
  if (!out || c < 0 || bootstrap_units < 1 || chunk_units < 1 || window_units < 0 || sink_units < 0)
    return SR_ERR_INVALID_ARG;
  const bool m = merge_single_frame_units != 0;
  const int64_t u0 = c == 0 ? 0 : bootstrap_units + static_cast<int64_t>(c - 1) * chunk_units;
  const int64_t nu = c == 0 ? bootstrap_units : chunk_units;
  const int64_t first = latents_before(u0, m);
  const int64_t n = latents_before(u0 + nu, m) - first;
  int64_t hist = 0;
  if (c > 0) {
    const int64_t hu = std::min<int64_t>(window_units, u0);
    hist = first - latents_before(u0 - hu, m);
  }
  const int64_t sink = latents_before(sink_units, m);
  const int64_t lim = INT32_MAX;
  if (first + n > lim || sink > lim) return SR_ERR_INVALID_ARG;
  out->first_frame = static_cast<int32_t>(first);
  out->n_frames = static_cast<int32_t>(n);
  out->hist_frames = static_cast<int32_t>(hist);
  out->sink_frames = static_cast<int32_t>(sink);
  return SR_OK;
}

// Cuts of one axis of n tokens into windows of `w` starting at offset `off`
// (a first window of off tokens when off > 0): the i-th window's start and size.
static int32_t axis_windows(int32_t n, int32_t w, int32_t off) { return off == 0 ? (n + w - 1) / w : 1 + (n - off + w - 1) / w; }
static void axis_window(int32_t n, int32_t w, int32_t off, int32_t i, int32_t& start, int32_t& size) {
  int32_t a, b;
  if (off == 0) {
    a = i * w;
    b = a + w;
  } else {
    a = i == 0 ? 0 : off + (i - 1) * w;
    b = i == 0 ? off : a + w;
  }
  start = a;
  size = std::min(b, n) - a;
}

static bool window_args_ok(int32_t gh, int32_t gw, int32_t window, int32_t shifted) {
  return gh >= 1 && gw >= 1 && window >= 2 && window <= 4096 && (shifted == 0 || shifted == 1) &&
         gh <= (1 << 20) && gw <= (1 << 20) && !(shifted && (window / 2 >= gh || window / 2 >= gw));
}

sr_status sr_window_count(int32_t grid_h, int32_t grid_w, int32_t window, int32_t shifted, int32_t* count) {
  if (!count || !window_args_ok(grid_h, grid_w, window, shifted)) return SR_ERR_INVALID_ARG;
  const int32_t off = shifted ? window / 2 : 0;
  *count = axis_windows(grid_h, window, off) * axis_windows(grid_w, window, off);
  return SR_OK;
}

sr_status sr_plan_window(int32_t grid_h, int32_t grid_w, int32_t window, int32_t shifted, int32_t index,
                         sr_window* out) {
  if (!out || !window_args_ok(grid_h, grid_w, window, shifted)) return SR_ERR_INVALID_ARG;
  const int32_t off = shifted ? window / 2 : 0;
  const int32_t nr = axis_windows(grid_h, window, off), nc = axis_windows(grid_w, window, off);
  if (index < 0 || index >= nr * nc) return SR_ERR_INVALID_ARG;
  axis_window(grid_h, window, off, index / nc, out->row0, out->rows);
  axis_window(grid_w, window, off, index % nc, out->col0, out->cols);
  return SR_OK;
}

sr_status sr_rope_angle(const sr_config* cfg, int32_t pair, int64_t position, float* angle) {
  if (!cfg || !angle) return SR_ERR_INVALID_ARG;
  sr_status st = validate_config(*cfg);
  if (st != SR_OK) return st;
  if (pair < 0 || pair >= cfg->head_dim / 2 || position <= -sr::kRopePositionLimit ||
      position >= sr::kRopePositionLimit)
    return SR_ERR_INVALID_ARG;
  sr::RopePhase ph;
  sr::rope_phase_table(cfg->rope_base, cfg->head_dim, &ph);
  *angle = sr::rope_angle(ph.turn_hi[pair], ph.turn_lo[pair], position, ph.rad_hi, ph.rad_lo);
  return SR_OK;
}

sr_status sr_session_free(sr_session* s) {
  delete s;
  return SR_OK;
}

sr_status sr_debug_wait_timeout(int32_t* err_word, uint64_t timeout_ns, void* stream) {
  if (!err_word || (reinterpret_cast<uintptr_t>(err_word) & 3u)) return SR_ERR_INVALID_ARG;
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return SR_ERR_INVALID_ARG;
  cudaError_t e = sr::launch_debug_wait(err_word, timeout_ns, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SR_OK : SR_ERR_CUDA;
}

}  // extern "C"
