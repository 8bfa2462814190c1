// attention.cu -- streaming chunk attention on the sm_103a tensor cores.
//
// O = softmax(scale * Q K^T) V for the chunk's queries over
//     sink bank[step]  U  visible ring frames  U  the chunk's own keys,
// with no mask: every chunk query sees every visible key, in both time
// directions (H3 project page, "Interactive Coding Worlds with Real-time
// Streaming Diffusion Render", section 3.1.2 and its "Prefix cache"
// paragraph, where the non-prefix rows see the whole window); each denoising
// step reads its own static-context bank (section 3.3 "Static-context KV
// caching"); cache slots that are still empty are simply not visited, so no
// mask is needed (section 3.2 Iteration 3 item 4, the seqused_k idea).
//
// A work unit = (session, head, block of 256 query rows). With a workspace
// the launch is persistent: one CTA per SM takes units from a launch-wide
// counter until none are left, and the producer loads the next unit's Q and
// first K/V while the softmax groups finish the current one. A full
// block is two 128-row tiles Q0, Q1 that share every K/V tile. The last block
// of a chunk may hold a single tile; then the two softmax groups take the two
// halves of the key range of that one tile ("split" mode) and merge their
// partial results at the end, so the tensor pipe still alternates between
// two independent score tiles. Units run longest first: every whole block
// (a last block of two tiles counts as whole), the blocks of one head side by
// side so that they read its keys and values through L2, then the single-tile
// last blocks. The kernel launches with programmatic stream serialization and
// touches no global memory before griddepcontrol.wait.
//
// Warp roles:
//   warps 0-3   softmax group 0 (thread i owns row i of its tile)
//   warps 4-7   softmax group 1
//   warp 8      MMA issuer (the whole warp in step, one elected lane issues):
//               tcgen05.mma, accumulators in TMEM
//   warp 9      TMA producer (one thread): Q once, then K/V tiles in stage
//               pairs (a K slot and a V slot behind one barrier), in the
//               order the MMA consumes them
//   warps 10-11 idle (they complete the third warpgroup)
//   warps 12-15 epilogue (head dim 128, two-tile units): read O_t out of TMEM
//               once its last PV MMAs are done, normalise it, stage the rows per
//               warp in shared memory and store them, while the softmax groups
//               already work on the next unit
// Registers: launched at 128 per thread (512 x 128 = 65536); the third and
// fourth warpgroups give back down to 80 and 64 and the two softmax warpgroups
// take 184 each: 2 x 128 x 184 + 128 x 80 + 128 x 64 = 65536, the launch's total.
// TMEM (512 columns): S0 [0,128) S1 [128,256) fp32 scores, O0 [256,256+d)
// O1 [384,384+d) fp32 accumulators. P (bf16) is written back over the first
// 64 columns of its S region and fed to the PV MMA straight from TMEM.
//
// Issue order of the MMA thread, i = iteration:
//   S0_0 S1_0 | PV0_0 S0_1 PV1_0 S1_1 | PV0_1 S0_2 PV1_1 S1_2 | ...
// so while softmax group 0 works on S0_i the tensor pipe runs PV1_{i-1} and
// S1_i, and the other way round. A softmax group hands its P over in two
// parts: the PV MMAs over the first keys start while it still converts the
// rest, and only the remainder of PV sits between its last P store and its
// next S. Online softmax in fp32 with exp2 and the
// scale folded into one packed FMA; the running maximum is only raised (and O
// rescaled in TMEM) when a new tile exceeds it by more than 2^8, which keeps
// numerator and denominator consistent and avoids most rescales.
#include <cuda_bf16.h>

#include <algorithm>

#include "sr_device.cuh"
#include "sr_kernels.h"

namespace sr {

namespace {

constexpr int BM = 128;      // rows per query tile
constexpr int BN = 128;      // keys per K/V tile
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kEpiWarp0 = 12;   // first warp of the epilogue warpgroup
constexpr int kLaunchRegs = 128;
constexpr uint32_t kRegsSoftmax = 184;
constexpr uint32_t kRegsOther = 80;
constexpr uint32_t kRegsEpi = 64;
static_assert(kEpiWarp0 * 32 + 128 == kAttnThreads, "the epilogue warpgroup is the last one");
static_assert(2 * 128 * kRegsSoftmax + 128 * (kRegsOther + kRegsEpi) <= kAttnThreads * kLaunchRegs,
              "register split exceeds what the block is launched with");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// P is handed to the PV MMAs in two parts: the first kPLoChunks 32-key chunks
// (p_half), then the rest (p_full).
constexpr int kPLoChunks = 2;

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;                 // 128-byte swizzle atoms per row
  static constexpr int kAtomBytes = BM * 128;           // one [128 rows][64 cols] bf16 box
  static constexpr int kTileBytes = kAtoms * kAtomBytes;
  // K/V ring depth. In split mode the second Q slot is free and serves as one
  // more stage (each iteration then needs four tiles: two K, two V).
  static constexpr int kStages = D == 128 ? 5 : 6;
  static constexpr int kStagesSplit = kStages + 1;
  // K/V travel in stage pairs (a K slot and a V slot behind one barrier)
  static constexpr int kPairs = kStages / 2;
  static constexpr int kPairsSplit = kStagesSplit / 2;
  static constexpr int kSmemQ = 2 * kTileBytes;
  static constexpr int kSmemKV = kStages * kTileBytes;
  static constexpr int kSmemBar = 2048;
  static constexpr int kSmemBytes = kSmemQ + kSmemKV + kSmemBar + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "more than 227 KB of shared memory per block");
  static constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, D, 1);
};

// Key tiles of a unit: segment s has nt[s] tiles over rows[s] valid rows,
// which start at row base[s] of its tensor map.
struct TileMap {
  int nt[kSegs];
  int rows[kSegs];
  int base[kSegs];
  __device__ __forceinline__ void locate(int j, int& seg, int& row0) const {
    seg = 0;
    while (seg < kSegs - 1 && j >= nt[seg]) {
      j -= nt[seg];
      ++seg;
    }
    row0 = j * BN;
  }
};

constexpr int kUnitSlots = 4;   // units published ahead by the producer (ring of records)

// One work unit as the producer decodes it; the MMA warp and the softmax
// groups read the record after the barrier that publishes it.
struct UnitRec {
  int u;                 // unit index; -1 once the CTA has no more work
  int si, head, part, parts;
  int q_local0;          // first query row of the unit (session-local)
  int q_row0, lq;        // the session's first row in the packed q / o, and its query rows
  int n_qtiles;          // 2 (shared mode) or 1 (split mode)
  int kv_lo, n_kv;       // the unit's range of the session's key tiles
  TileMap tm;
};

struct SmemBars {
  uint64_t q_full;
  uint64_t q_empty;       // the unit's QK MMAs are done: both Q slots may be reloaded
  uint64_t kv_full[8];    // shared-mode pairs at [0, kPairs), split-mode pairs at [4, 4 + kPairsSplit)
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_half[2];     // group t has stored the first kPLoChunks chunks of P_t
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t unit_ready[kUnitSlots];
  uint64_t x_full;        // split mode: group 1 has published its running max and sum
  uint64_t x_empty;       // split mode: group 0 has read them and both O accumulators
  uint64_t part_done;     // key split: group 0's partial rows are published
  uint64_t part_last;     // key split: `last` is set
  uint64_t drain;
  uint64_t il_full[2];    // two-tile unit: softmax group t has published 1/l of its rows
  uint64_t il_free[2];    // the epilogue warpgroup has read them
  uint64_t o_free[2];     // the epilogue warpgroup has read O_t: the next PV may overwrite it
  uint32_t tmem_base;
  int abort;
  int last;       // key-split last block: this CTA is the last part and merges
  int stage_done; // epilogue warps done with a unit's staging (4 per two-tile unit)
  // split mode: group 1's running max / sum, handed to group 0; two-tile unit:
  // 1/l of tile 0 (xm) and tile 1 (xl), handed to the epilogue warpgroup
  float xm[BM];
  float xl[BM];
  UnitRec rec[kUnitSlots];
};

// The last part of a key-split last block combines every part's published
// fp32 rows (O and the log2-sum-exp in column D of [part][128][D + 4]) into
// bf16 output rows and their natural-log LSE. Warp w of the merging group
// takes rows w, w + 4, ... and each lane D/32 columns of them, so that a load
// or store of a row is one contiguous access of the warp, and the loads of all
// parts of kMergeRows rows are in flight together. Out of line: it runs once per
// last block and keeps its registers out of the softmax loop's allocation.
template <int D>
__device__ __noinline__ void merge_key_parts(const float* __restrict__ hbase, int parts, int n_live,
                                             __nv_bfloat16* __restrict__ o, int n_heads, int head, int64_t row0,
                                             float* __restrict__ lse, int64_t lse_ld, int w, int lane) {
  __threadfence();
  constexpr int kCpl = D / 32;   // columns per lane
  constexpr int kMergeRows = 4;
  const int64_t pstride = static_cast<int64_t>(BM) * (D + 4);
#pragma unroll 1
  for (int rb = w; rb < n_live; rb += 4 * kMergeRows) {
    float lw[kMergeRows][kMaxTailSplit];
    float x[kMergeRows][kMaxTailSplit][kCpl];
#pragma unroll
    for (int q = 0; q < kMergeRows; ++q) {
      const int rr = min(rb + 4 * q, n_live - 1);   // a row past the end repeats the last one
#pragma unroll
      for (int k = 0; k < kMaxTailSplit; ++k) {
        lw[q][k] = -INFINITY;
        if (k < parts) {
          const float* src = hbase + k * pstride + static_cast<int64_t>(rr) * (D + 4);
          lw[q][k] = __ldcg(src + D);
          if constexpr (kCpl == 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src) + lane);
            x[q][k][0] = v.x; x[q][k][1] = v.y; x[q][k][2] = v.z; x[q][k][3] = v.w;
          } else {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(src) + lane);
            x[q][k][0] = v.x; x[q][k][1] = v.y;
          }
        } else {
#pragma unroll
          for (int c = 0; c < kCpl; ++c) x[q][k][c] = 0.f;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kMergeRows; ++q) {
      const int rr = rb + 4 * q;
      if (rr < n_live) {
        float mx = lw[q][0];
#pragma unroll
        for (int k = 1; k < kMaxTailSplit; ++k) mx = fmaxf(mx, lw[q][k]);
        float L = 0.f;
        float a[kCpl];
#pragma unroll
        for (int c = 0; c < kCpl; ++c) a[c] = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxTailSplit; ++k) {
          const float wk = ex2_approx(lw[q][k] - mx);   // 0 for an absent part
          L += wk;
#pragma unroll
          for (int c = 0; c < kCpl; ++c) a[c] = fmaf(wk, x[q][k][c], a[c]);
        }
        const float invL = 1.f / L;
        __nv_bfloat16* dst = o + ((row0 + rr) * n_heads + head) * D + lane * kCpl;
        if constexpr (kCpl == 4) {
          uint2 pk;
          pk.x = pack_bf16x2(a[0] * invL, a[1] * invL);
          pk.y = pack_bf16x2(a[2] * invL, a[3] * invL);
          *reinterpret_cast<uint2*>(dst) = pk;
        } else {
          *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(a[0] * invL, a[1] * invL);
        }
        if (lane == 0 && lse != nullptr)
          lse[static_cast<int64_t>(head) * lse_ld + row0 + rr] = (mx + __log2f(L)) * 0.69314718055994531f;
      }
    }
  }
}

// The key tiles each query tile walks, within the unit's range [lo, lo + n) of
// all key tiles: in shared mode both walk the whole range; in split mode tile 0
// walks [lo, lo + h) and tile 1 walks [lo + h, lo + n).
struct Walk {
  bool split;
  int lo, n, h;
  __device__ __forceinline__ int count(int t) const { return split ? (t == 0 ? h : n - h) : n; }
  __device__ __forceinline__ int kv(int t, int i) const { return lo + ((split && t == 1) ? h + i : i); }
  __device__ __forceinline__ int iters() const { return split ? h : n; }
};

template <int NSESS>
__device__ __forceinline__ void decode_unit(const AttnParams<NSESS>& p, int u, int H, int& si, int& head,
                                            int& qb, int& part, int& tile) {
  part = 0;
  si = 0;
  tile = -1;   // the unit is a whole block or a last block
  const int n_whole = p.n_full_units - p.n_conv;
  if (u < n_whole) {
    // whole blocks, session by session, the blocks of one head next to each
    // other (they read the same keys and values, which then come from L2)
#pragma unroll 1
    while (si + 1 < p.n_sess && u >= p.whole_end[si]) ++si;
    const int local = u - p.sess[si].unit_begin;
    const int nf = p.sess[si].nfull;
    head = local / nf;
    qb = local % nf;
  } else if (u < p.n_full_units + p.n_conv) {
    // the last n_conv whole blocks, two single-tile units each
    const int v = u - n_whole;
    const int b = n_whole + v / 2;
    tile = v % 2;
#pragma unroll 1
    while (si + 1 < p.n_sess && b >= p.whole_end[si]) ++si;
    const int local = b - p.sess[si].unit_begin;
    const int nf = p.sess[si].nfull;
    head = local / nf;
    qb = local % nf;
  } else {
    // single-tile last blocks (H per session that has them), each run as
    // tail_split key-range parts
    const int t = u - p.n_full_units - p.n_conv;
    const int tail = t / p.tail_split;
    part = t - tail * p.tail_split;
#pragma unroll 1
    while (si + 1 < p.n_sess && tail >= p.tail_end[si]) ++si;
    head = tail - p.sess[si].tail_begin;
    qb = p.sess[si].nqb - 1;
  }
}

// Decode unit u into its record: session, head, query block and key range,
// and the tile map of its key segments (from the device frame counter for a
// device-state call).
template <int NSESS>
__device__ __forceinline__ void make_unit(const AttnParams<NSESS>& p, int u, UnitRec& r) {
  int si, head, qb, part, tile;
  decode_unit(p, u, p.n_heads, si, head, qb, part, tile);
  const AttnSession& S = p.sess[si];
  TileMap tl;
#pragma unroll
  for (int s = 0; s < kSegs; ++s) {
    tl.rows[s] = S.seg_rows[s];
    tl.base[s] = 0;
  }
  if (S.dev_n != nullptr) {
    // The visible ring frames follow the device frame counter: frames n-h ..
    // n-1 in slots (g mod W), one or two row ranges of the whole-ring maps.
    const int64_t n = *S.dev_n;
    const int W = S.ring_W, T = S.ring_T;
    const int v = static_cast<int>(min(n, static_cast<int64_t>(W)));
    const int h = S.hist_req < 0 ? v : min(S.hist_req, v);
    if (h == W) {
      tl.rows[1] = W * T;
      tl.rows[2] = 0;
    } else if (h > 0) {
      const int start = static_cast<int>((n - h) % W);
      const int a = min(h, W - start);
      tl.base[1] = start * T;
      tl.rows[1] = a * T;
      tl.rows[2] = (h - a) * T;
    } else {
      tl.rows[1] = tl.rows[2] = 0;
    }
  }
  int n_kv_all = 0;
#pragma unroll
  for (int s = 0; s < kSegs; ++s) {
    tl.nt[s] = (tl.rows[s] + BN - 1) / BN;
    n_kv_all += tl.nt[s];
  }
  r.si = si;
  r.head = head;
  r.part = part;
  r.q_local0 = qb * 2 * BM + (tile > 0 ? BM : 0);
  r.n_qtiles = tile >= 0 ? 1 : min(2, (S.lq - r.q_local0 + BM - 1) / BM);
  r.q_row0 = S.q_row0;
  r.lq = S.lq;
  // a single-tile last block may be one of `parts` units sharing its key range
  r.parts = (tile < 0 && r.n_qtiles == 1 && S.ws_part != nullptr) ? p.tail_split : 1;
  r.kv_lo = static_cast<int>(static_cast<int64_t>(part) * n_kv_all / r.parts);
  r.n_kv = static_cast<int>(static_cast<int64_t>(part + 1) * n_kv_all / r.parts) - r.kv_lo;
  r.tm = tl;
  r.u = u;
}

__device__ __forceinline__ Walk unit_walk(const UnitRec& r) {
  const bool split = r.n_qtiles == 1;
  return Walk{split, r.kv_lo, r.n_kv, split ? (r.n_kv + 1) / 2 : r.n_kv};
}

// The unit a CTA takes after its first (which is its block index): the next
// one of a launch-wide counter, or none when the launch runs one unit per
// CTA. The counter holds (epoch << 32 | units taken); raising it to this
// call's epoch first discards a count left by an earlier call that stopped
// early. The last CTA to run out of units clears it (and the count of CTAs
// that ran out), so that a replay of the same launch starts from zero.
template <int NSESS>
__device__ __forceinline__ int next_unit(const AttnParams<NSESS>& p, bool& tagged) {
  if (p.unit_ctr == nullptr) return p.n_units;
  const unsigned long long tag = static_cast<unsigned long long>(p.epoch) << 32;
  if (!tagged) {   // once this CTA has raised it, the counter carries this call's epoch
    atomicMax(p.unit_ctr, tag);
    tagged = true;
  }
  const unsigned long long old = atomicAdd(p.unit_ctr, 1ull);
  const int u = static_cast<int>(gridDim.x + (old & 0xffffffffull));
  if (u >= p.n_units) {
    atomicMax(p.unit_ctr + 1, tag);
    const unsigned long long d = atomicAdd(p.unit_ctr + 1, 1ull);
    if ((d & 0xffffffffull) == gridDim.x - 1) {
      atomicExch(p.unit_ctr, 0ull);
      atomicExch(p.unit_ctr + 1, 0ull);
    }
  }
  return u;
}

template <int D, int NSESS>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams<NSESS> p) {
  using C = Cfg<D>;
  static_assert(sizeof(SmemBars) <= C::kSmemBar, "barrier area too small");
  // The previous kernel of the stream may still be draining: the set-up below
  // touches no global memory until grid_dep_wait(). The next kernel may be
  // scheduled as soon as every CTA of this grid has started.
  grid_dep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::kSmemQ;
  SmemBars* bars = reinterpret_cast<SmemBars*>(smem + C::kSmemQ + C::kSmemKV);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  WaitCtx wc{&bars->abort, p.err_word, p.timeout_ns};

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < 8; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_half[t], BM);
      mbar_init(&bars->p_full[t], BM);
      mbar_init(&bars->o_done[t], 1);
    }
    for (int k = 0; k < kUnitSlots; ++k) mbar_init(&bars->unit_ready[k], 1);
    mbar_init(&bars->x_full, BM);
    mbar_init(&bars->x_empty, BM);
    mbar_init(&bars->part_done, BM);
    mbar_init(&bars->part_last, 1);
    mbar_init(&bars->drain, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->il_full[t], BM);
      mbar_init(&bars->il_free[t], BM);
      mbar_init(&bars->o_free[t], BM);
    }
    bars->abort = 0;
    bars->stage_done = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();
  const uint32_t tmem = bars->tmem_base;

  // Work: this CTA's first unit is its block index; a persistent launch (one
  // CTA per SM) then takes further units from the launch-wide counter. Each
  // role walks the same sequence of units: the producer decodes a unit into
  // bars->rec[k % kUnitSlots] and publishes it on unit_ready (the softmax
  // groups and the epilogue warpgroup) and q_full (the MMA warp). A slot is
  // reused four units later: by then the MMA warp has waited for the epilogue
  // warpgroup to read out at least unit k - 3, after it read that record.
  // Every barrier keeps running phase counts across units.
  if (warp >= kEpiWarp0) {
    regs_dec<kRegsEpi>();
    if constexpr (D == 128) {
      // ------------------------------------------------------------ epilogue
      // Two-tile units only (the softmax groups keep the others). Per tile t:
      // take 1/l of its rows from the softmax group, wait for the last PV MMAs
      // into O_t, read O_t out of TMEM (scaled, rounded to bf16) into this
      // warp's 32 rows of the fifth K/V stage, which two-tile units leave
      // unused, release O_t to the next unit's PV MMAs, then store the rows so
      // that 16 lanes write each 256-byte row whole. 16-byte chunk j of staged
      // row rr sits at rr * 256 + ((j & 8) | ((j ^ rr) & 7)) * 16: neither the
      // row-per-lane writes nor the two-rows-per-instruction reads conflict on
      // banks.
      const int eq = warp % 4;   // TMEM lane quarter: rows 32 eq .. 32 eq + 31 of each tile
      const uint32_t lane_base = static_cast<uint32_t>(eq * 32) << 16;
      constexpr int kRowBytes = D * 2;
      uint8_t* stg = sKV + 4 * C::kTileBytes + eq * 32 * kRowBytes;
      bool ok = true;
      int uk = 0;
      uint32_t od0 = 0, od1 = 0;   // o_done completions of each tile so far
      uint32_t nw = 0;             // two-tile units so far
      while (ok) {
        ok = __all_sync(0xffffffffu, wait_bounded(&bars->unit_ready[uk % kUnitSlots], (uk / kUnitSlots) & 1, wc, 12));
        if (!ok) break;
        const UnitRec& r = bars->rec[uk % kUnitSlots];
        if (r.u < 0) break;
        const bool split = r.n_qtiles == 1;
        const uint32_t w0 = od0, w1 = od1;
        od0 += 1u;
        od1 += (!split || r.n_kv - (r.n_kv + 1) / 2 > 0) ? 1u : 0u;   // as the softmax groups count
        ++uk;
        if (split) continue;
        const int head = r.head;
        const int64_t row0 = static_cast<int64_t>(r.q_row0) + r.q_local0 + eq * 32;
        const int live0 = r.lq - r.q_local0 - eq * 32;
        for (int t = 0; t < 2 && ok; ++t) {
          ok = __all_sync(0xffffffffu, wait_bounded(&bars->il_full[t], nw & 1u, wc, 13));
          if (!ok) break;
          const float inv = (t == 0 ? bars->xm : bars->xl)[eq * 32 + lane];
          mbar_arrive(&bars->il_free[t]);
          ok = __all_sync(0xffffffffu, wait_bounded(&bars->o_done[t], (t == 0 ? w0 : w1) & 1u, wc, 14));
          if (!ok) break;
          tc_fence_after();
          const uint32_t t_o = tmem + lane_base + 256 + t * 128;
          uint8_t* mine = stg + lane * kRowBytes;
#pragma unroll 1
          for (int q = 0; q < D / 16; ++q) {
            uint32_t o[16];
            tmem_ld16(t_o + q * 16, o);
            tmem_wait_ld();
            tmem_fix(o);
            uint4 pk[2];
            uint32_t* w = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int j = 2 * q + h;
              *reinterpret_cast<uint4*>(mine + ((j & 8) | ((j ^ lane) & 7)) * 16) = pk[h];
            }
          }
          // O_t is read: the next unit's PV MMAs may overwrite it
          tc_fence_before();
          mbar_arrive(&bars->o_free[t]);
          __syncwarp();
          const int live = live0 - t * BM;
          const int64_t ld = static_cast<int64_t>(p.n_heads) * D;
          __nv_bfloat16* orow = p.o + (row0 + t * BM) * ld + head * D;
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const int rr = 2 * i + lane / 16, j = lane % 16;
            const uint4 v = *reinterpret_cast<const uint4*>(stg + rr * kRowBytes + ((j & 8) | ((j ^ rr) & 7)) * 16);
            if (rr < live) *reinterpret_cast<uint4*>(orow + rr * ld + j * 8) = v;
          }
          __syncwarp();
        }
        ++nw;
        // the stage may next be filled by a tensor copy (a single-tile unit)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          atomicAdd(&bars->stage_done, 1);
        }
      }
    }
  } else if (warp >= 8) {
    regs_dec<kRegsOther>();
    if (warp == kTmaWarp && lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      tma_prefetch_map(&p.qmap);
      bool ok = true;
      int uk = 0;            // units of this CTA so far
      int u = blockIdx.x;
      int q_last = -1;       // the last unit whose Q load was issued
      int q_shared = 0, q_split = 0;   // pair loads issued so far, per mode
      int mode = -1;         // the previous unit's mode
      uint32_t nwg = 0;      // two-tile units (head dim 128) issued: their rows are staged in the fifth stage
      auto slot_ptr = [&](int slot) -> uint8_t* {
        return slot < C::kStages ? sKV + slot * C::kTileBytes : sQ + C::kTileBytes;
      };
      // Publish unit k's record (or the end of work) for the softmax groups.
      // The record of the next unit goes out as soon as this unit's loads are
      // issued, so that the softmax groups find it when they finish this
      // unit's epilogue; its slot was last used four units back.
      auto publish = [&](int k, int unit) {
        UnitRec& rk = bars->rec[k % kUnitSlots];
        if (unit >= p.n_units)
          rk.u = -1;
        else
          make_unit(p, unit, rk);
        mbar_arrive(&bars->unit_ready[k % kUnitSlots]);
      };
      bool tagged = false;
      publish(0, u);
      while (ok) {
        // both Q slots (and the split-mode stage in the second) are free once
        // the previous unit's MMAs that read them are done
        if (uk > 0 && !wait_bounded(&bars->q_empty, (uk - 1) & 1, wc, 7)) {
          ok = false;
          break;
        }
        const UnitRec& r = bars->rec[uk % kUnitSlots];
        if (r.u < 0) {
          mbar_arrive(&bars->q_full);
          break;
        }
        const AttnSession& S = p.sess[r.si];
        const TileMap& tm = r.tm;
        const Walk wk = unit_walk(r);
        const int md = wk.split ? 1 : 0;
        // K/V travel in stage pairs behind one barrier: pair p is the slots
        // 2p (a K tile) and 2p+1 (a V tile); the extra split-mode slot is the
        // second Q slot. The two modes use separate barriers over the same
        // slots, so on a change of mode the previous mode's pairs must have
        // been released first.
        if (mode >= 0 && mode != md) {
          const int np = mode ? C::kPairsSplit : C::kPairs;
          const int b0 = mode ? 4 : 0;
          const int qm = mode ? q_split : q_shared;
          for (int k = max(0, qm - np); k < qm && ok; ++k)
            ok = wait_bounded(&bars->kv_empty[b0 + k % np], (k / np) & 1, wc, 1);
          // split mode also loads into the fifth stage, where the epilogue
          // warpgroup stages output rows: wait until it is done with every
          // two-tile unit so far (four warps count each)
          if (ok && md == 1 && D == 128 && nwg > 0) ok = wait_count(&bars->stage_done, static_cast<int>(4 * nwg), wc, 16);
          if (!ok) break;
        }
        mode = md;
        for (int s = 0; s < kSegs; ++s)
          if (tm.nt[s]) {
            tma_prefetch_map(&S.kmap[s]);
            tma_prefetch_map(&S.vmap[s]);
          }
        mbar_arrive_expect_tx(&bars->q_full, r.n_qtiles * C::kTileBytes);
        for (int t = 0; t < r.n_qtiles; ++t)
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_2d(sQ + t * C::kTileBytes + a * C::kAtomBytes, &p.qmap, &bars->q_full,
                        r.head * D + a * 64, r.q_row0 + r.q_local0 + t * BM, pol_q);
        q_last = uk;
        const int npair = md ? C::kPairsSplit : C::kPairs;
        const int bar0 = md ? 4 : 0;
        int q = md ? q_split : q_shared;
        auto issue = [&](int j, bool is_v, int slot, uint64_t* bar) {
          int seg, row0;
          tm.locate(j, seg, row0);
          const CUtensorMap* map = is_v ? &S.vmap[seg] : &S.kmap[seg];
          uint8_t* dst = slot_ptr(slot);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_2d(dst + a * C::kAtomBytes, map, bar, r.head * D + a * 64, tm.base[seg] + row0, pol_kv);
        };
        // one pair: key tile kj (if >= 0) and value tile vj (if >= 0)
        auto load_pair = [&](int kj, int vj) {
          if (!ok) return;
          const int pr = q % npair;
          if (q >= npair && !wait_bounded(&bars->kv_empty[bar0 + pr], ((q / npair) - 1) & 1, wc, 1)) {
            ok = false;
            return;
          }
          uint64_t* bar = &bars->kv_full[bar0 + pr];
          mbar_arrive_expect_tx(bar, ((kj >= 0 ? 1 : 0) + (vj >= 0 ? 1 : 0)) * C::kTileBytes);
          if (kj >= 0) issue(kj, false, 2 * pr, bar);
          if (vj >= 0) issue(vj, true, 2 * pr + 1, bar);
          ++q;
        };
        const int n_it = wk.iters();
        if (!wk.split) {
          // shared mode, iteration i: K_i (the S MMAs of both tiles) and V_{i-1}
          for (int i = 0; i <= n_it && ok; ++i) load_pair(i < n_it ? i : -1, i > 0 ? i - 1 : -1);
        } else {
          // split mode, iteration i and tile t: K(t, i) and V(t, i-1), tile 0 first
          for (int i = 0; i <= n_it && ok; ++i)
            for (int t = 0; t < 2; ++t) {
              const bool kq = i < wk.count(t), vq = i > 0 && i - 1 < wk.count(t);
              if (kq || vq) load_pair(kq ? wk.kv(t, i) : -1, vq ? wk.kv(t, i - 1) : -1);
            }
        }
        if (md)
          q_split = q;
        else
          q_shared = q;
        if (D == 128 && !md) ++nwg;
        if (!ok) break;
        u = next_unit(p, tagged);   // taken once this unit's loads are all issued
        publish(uk + 1, u);
        ++uk;
      }
      if (!ok || bars->abort) {
        // let every copy this CTA started land before shared memory is released
        if (q_last >= 0) wait_drain(&bars->q_full, q_last & 1, p.timeout_ns);
        if (mode >= 0) {
          const int np = mode ? C::kPairsSplit : C::kPairs;
          const int b0 = mode ? 4 : 0;
          const int qm = mode ? q_split : q_shared;
          for (int k = max(0, qm - np); k < qm; ++k)
            wait_drain(&bars->kv_full[b0 + k % np], (k / np) & 1, p.timeout_ns);
        }
      }
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp runs this loop in step; one elected lane issues the
      // MMAs and commits. Keeping the warp converged lets the descriptor and
      // loop arithmetic run warp-uniform instead of as one divergent thread.
      const uint32_t leader = elect_one();
      bool issued_any = false;
      bool ok = true;
      const uint32_t sq = smem_u32(sQ);
      const uint32_t skv = smem_u32(sKV);
      int uk = 0;
      // Position in the producer's sequence of stage pairs, per mode: pair and
      // phase parity of the next one, advanced by counters (no division here).
      int pc_shared = 0, pc_split = 0;
      uint32_t ph_shared = 0, ph_split = 0;
      uint32_t pb0 = 0, pb1 = 0;   // P tiles of each softmax group waited on so far
      uint32_t nwg = 0;            // two-tile units whose O the epilogue warpgroup reads out
      bool prev_wg = false;        // the previous unit was one of them
      // shared-memory address of a K/V stage (the extra split-mode stage is the second Q slot)
      auto stage_addr = [&](int stage) -> uint32_t {
        return stage < C::kStages ? skv + stage * C::kTileBytes : sq + C::kTileBytes;
      };
      while (ok) {
        ok = __all_sync(0xffffffffu, wait_bounded(&bars->q_full, uk & 1, wc, 2));
        if (!ok) break;
        const UnitRec& r = bars->rec[uk % kUnitSlots];
        if (r.u < 0) break;
        const Walk wk = unit_walk(r);
        const int md = wk.split ? 1 : 0;
        const int npair = md ? C::kPairsSplit : C::kPairs;
        const int bar0 = md ? 4 : 0;
        int pc = md ? pc_split : pc_shared;
        uint32_t ph = md ? ph_split : ph_shared;
        auto take = [&]() -> int {   // wait for the next pair; returns its index
          const int p0 = pc;
          if (ok) ok = __all_sync(0xffffffffu, wait_bounded(&bars->kv_full[bar0 + p0], ph, wc, 3));
          if (++pc == npair) {
            pc = 0;
            ph ^= 1u;
          }
          return p0;
        };
        // softmax group t has written the first part (half) or all of P_t of iteration it
        auto wait_p = [&](int t, int it, bool half) {
          const uint32_t par = ((t == 0 ? pb0 : pb1) + static_cast<uint32_t>(it)) & 1u;
          if (ok) ok = __all_sync(0xffffffffu, wait_bounded(half ? &bars->p_half[t] : &bars->p_full[t], par, wc,
                                                            half ? 14 : 4));
          tc_fence_after();
        };
        auto qk = [&](int t, int stage) {   // S_t = Q_t K^T
          const uint32_t d_tmem = tmem + t * BN;
          const uint32_t qt = sq + (wk.split ? 0 : t) * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::kAtomBytes + (kk % 4) * 32;
            const uint64_t ad = sdesc_sw128(qt + off, 16, 1024);
            const uint64_t bd = sdesc_sw128(stage_addr(stage) + off, 16, 1024);
            mma_ss_w(d_tmem, ad, bd, C::kIdescS, kk > 0 ? 1u : 0u, leader);
          }
        };
        // O_t += P_t V over key steps [k0, k1) of 16 keys
        auto pv_part = [&](int t, int stage, bool acc, int k0, int k1) {
          const uint32_t d_tmem = tmem + 256 + t * 128;
          const uint32_t a_tmem = tmem + t * BN;
#pragma unroll
          for (int kk = k0; kk < k1; ++kk) {
            const uint64_t bd = sdesc_sw128(stage_addr(stage) + kk * 16 * 128, C::kAtomBytes, 1024);
            mma_ts_w(d_tmem, a_tmem + kk * 8, bd, C::kIdescPV, (acc || kk > 0) ? 1u : 0u, leader);
          }
        };
        // The epilogue warpgroup has read O_t of the previous unit: the unit's
        // first PV MMA into O_t may overwrite it.
        auto free_o = [&](int t) {
          if (prev_wg && ok) ok = __all_sync(0xffffffffu, wait_bounded(&bars->o_free[t], (nwg - 1) & 1u, wc, 15));
          tc_fence_after();
        };
        // O_t += P_t V of iteration it, each part of P as soon as it is stored
        auto pv = [&](int t, int stage, bool acc, int it) {
          wait_p(t, it, true);
          if (!ok) return;
          pv_part(t, stage, acc, 0, 2 * kPLoChunks);
          wait_p(t, it, false);
          if (!ok) return;
          pv_part(t, stage, acc, 2 * kPLoChunks, BN / 16);
        };
        if (!wk.split) {
          // Shared mode: both tiles walk all n key tiles, and the loop carries
          // nothing between two MMA bursts but the waits it cannot avoid. The
          // tensor pipe queues only a few MMAs, so every cycle of other work
          // between bursts (a division, a loop back edge, a branch) is a cycle
          // the pipe may stand idle: stages advance by counters and the first
          // and last iterations are peeled off, so the body branches only to
          // leave on an abort.
          const int n = wk.n;
          // iteration 0: S_0 of both tiles (pair 0 holds K_0 only)
          const int p0 = take();
          if (ok) {
            tc_fence_after();
            qk(0, 2 * p0);
            tc_commit_w(&bars->s_full[0], leader);
            qk(1, 2 * p0);
            tc_commit_w(&bars->s_full[1], leader);
            tc_commit_w(&bars->kv_empty[bar0 + p0], leader);
            issued_any = true;
          }
          // iterations 1 .. n-1: PV_{i-1} and S_i of both tiles from one pair
          // (K_i, V_{i-1}). Its wait comes first, while the warp would otherwise
          // be waiting for softmax group 0; between S0_i and PV1_{i-1} there is
          // only that group's wait. Iteration 1 holds the unit's first PV of
          // each tile, which may have to wait until O_t is read out: peeled.
          if (n > 1 && ok) {
            const int pi = take();
            tc_fence_after();
            free_o(0);
            pv(0, 2 * pi + 1, false, 0);
            if (ok) {
              qk(0, 2 * pi);
              tc_commit_w(&bars->s_full[0], leader);
              free_o(1);
              pv(1, 2 * pi + 1, false, 0);
            }
            if (ok) {
              qk(1, 2 * pi);
              tc_commit_w(&bars->s_full[1], leader);
              tc_commit_w(&bars->kv_empty[bar0 + pi], leader);
            }
          }
          for (int i = 2; i < n && ok; ++i) {
            const int pi = take();
            tc_fence_after();
            pv(0, 2 * pi + 1, i > 1, i - 1);
            if (!ok) break;
            qk(0, 2 * pi);
            tc_commit_w(&bars->s_full[0], leader);
            pv(1, 2 * pi + 1, i > 1, i - 1);
            if (!ok) break;
            qk(1, 2 * pi);
            tc_commit_w(&bars->s_full[1], leader);
            tc_commit_w(&bars->kv_empty[bar0 + pi], leader);
          }
          // every S MMA of the unit is issued: the Q slots free up as they finish
          if (ok) tc_commit_w(&bars->q_empty, leader);
          // last: PV_{n-1} of both tiles (the last pair holds V_{n-1} only)
          if (ok) {
            const int pl = take();
            tc_fence_after();
            if (ok && n == 1) free_o(0);
            if (ok) pv(0, 2 * pl + 1, n > 1, n - 1);
            if (ok) {
              tc_commit_w(&bars->o_done[0], leader);
              if (n == 1) free_o(1);
              if (ok) pv(1, 2 * pl + 1, n > 1, n - 1);
            }
            if (ok) {
              tc_commit_w(&bars->o_done[1], leader);
              tc_commit_w(&bars->kv_empty[bar0 + pl], leader);
            }
          }
        } else {
          // Split mode (a single-tile last block): tile 0 walks c0 key tiles,
          // tile 1 the next c1 (c0 - c1 is 0 or 1). Iteration i takes, per tile
          // t, one pair holding K(t, i) and V(t, i-1); tile 1's wait comes after
          // tile 0's MMAs are queued.
          const int c0 = wk.count(0), c1 = wk.count(1);
          free_o(0);
          free_o(1);
          for (int i = 0; i <= c0 && ok; ++i) {
            const bool p0 = i > 0 && i - 1 < c0, q0 = i < c0;
            if (p0 || q0) {
              const int pr = take();   // K(0, i) and V(0, i-1)
              if (!ok) break;
              tc_fence_after();
              if (p0) {
                pv(0, 2 * pr + 1, i > 1, i - 1);
                if (!ok) break;
                if (i == c0) tc_commit_w(&bars->o_done[0], leader);
              }
              if (q0) {
                qk(0, 2 * pr);
                tc_commit_w(&bars->s_full[0], leader);
                issued_any = true;
              }
              tc_commit_w(&bars->kv_empty[bar0 + pr], leader);
            }
            const bool p1 = i > 0 && i - 1 < c1, q1 = i < c1;
            if (p1 || q1) {
              const int pr = take();   // K(1, i) and V(1, i-1)
              if (!ok) break;
              tc_fence_after();
              if (p1) {
                pv(1, 2 * pr + 1, i > 1, i - 1);
                if (!ok) break;
                if (i == c1) tc_commit_w(&bars->o_done[1], leader);
              }
              if (q1) {
                qk(1, 2 * pr);
                tc_commit_w(&bars->s_full[1], leader);
              }
              tc_commit_w(&bars->kv_empty[bar0 + pr], leader);
            }
          }
          // the second Q slot served as a K/V stage: free once every MMA is done
          if (ok) tc_commit_w(&bars->q_empty, leader);
        }
        if (md) {
          pc_split = pc;
          ph_split = ph;
        } else {
          pc_shared = pc;
          ph_shared = ph;
        }
        pb0 += static_cast<uint32_t>(wk.count(0));
        pb1 += static_cast<uint32_t>(wk.count(1));
        prev_wg = D == 128 && !wk.split;
        if (prev_wg) ++nwg;
        ++uk;
      }
      if (!ok && issued_any) {
        // no tensor-core work may still be running when TMEM is released
        tc_commit_w(&bars->drain, leader);
        wait_drain(&bars->drain, 0, p.timeout_ns);
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax groups
    const int t = warp / 4;
    const int row = threadIdx.x % BM;
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + t * BN;
    const uint32_t t_o = tmem + lane_base + 256 + t * 128;
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    bool ok = true;
    int uk = 0;
    uint32_t sb = 0;             // S tiles of this group consumed so far
    uint32_t od0 = 0, od1 = 0;   // o_done completions of each tile so far
    uint32_t nx = 0;             // split-mode units so far
    uint32_t nk = 0;             // key-split units so far
    uint32_t nwg = 0;            // two-tile units handed to the epilogue warpgroup
    uint32_t nwg_seen = 0;       // of those, known to be finished by it
    while (ok) {
      ok = __all_sync(0xffffffffu, wait_bounded(&bars->unit_ready[uk % kUnitSlots], (uk / kUnitSlots) & 1, wc, 8));
      if (!ok) break;
      const UnitRec& r = bars->rec[uk % kUnitSlots];
      if (r.u < 0) break;
      const Walk wk = unit_walk(r);
      const TileMap& tm = r.tm;
      const AttnSession& S = p.sess[r.si];
      const int head = r.head, part = r.part, parts = r.parts;
      float m = -INFINITY;   // running max of scaled scores, log2 units
      float l = 0.f;         // running sum of exp2(score - m)
      const int cnt = wk.count(t);
      for (int j = 0; ok && j < cnt; ++j) {
        // ragged tail of a segment: keys past its end are not part of the window.
        // Looked up before the wait, so the shared-memory latency hides behind it.
        int seg, row0;
        tm.locate(wk.kv(t, j), seg, row0);
        const int valid = tm.rows[seg] - row0;
        ok = wait_bounded(&bars->s_full[t], (sb + static_cast<uint32_t>(j)) & 1u, wc, 5);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t rr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, rr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_fix(rr[c]);
        float* s = reinterpret_cast<float*>(&rr[0][0]);
        if (valid < BN) {
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (i >= valid) s[i] = -INFINITY;
        }
        float a0 = fmaxf(s[0], s[1]), a1 = fmaxf(s[2], s[3]), a2 = fmaxf(s[4], s[5]), a3 = fmaxf(s[6], s[7]);
#pragma unroll
        for (int i = 8; i < BN; i += 8) {
          a0 = fmax3(a0, s[i], s[i + 1]);
          a1 = fmax3(a1, s[i + 2], s[i + 3]);
          a2 = fmax3(a2, s[i + 4], s[i + 5]);
          a3 = fmax3(a3, s[i + 6], s[i + 7]);
        }
        const float mt = fmax3(a0, a1, fmaxf(a2, a3)) * sl2;
        const bool need = (j == 0) || (mt > m + kRescaleThreshold);
        float f = 1.f;                    // factor that takes O and l to the new maximum
        const bool rescale = __any_sync(0xffffffffu, need);
        if (rescale) {
          const float m_new = fmaxf(m, mt);
          if (j > 0) f = ex2_approx(m - m_new);
          m = m_new;
        }
        const float2 negm = make_float2(-m, -m);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int i = c * 32 + 2 * k;
            const float2 x = __ffma2_rn(make_float2(s[i], s[i + 1]), sl2x2, negm);
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            acc[k % 4] = __fadd2_rn(acc[k % 4], e);
            pk[k] = pack_bf16x2(e.x, e.y);
          }
          tmem_st16(t_s + c * 16, pk);
          if (c == kPLoChunks - 1) {
            if (rescale && j > 0) {
              // O was last written by PV_{j-1}, which completed before S_j was
              // signalled (in-order tensor pipe; a commit covers all prior
              // MMAs); no MMA of PV_j is issued before this thread arrives on
              // p_half. Done here, where the scores of the chunks already
              // converted no longer hold registers.
#pragma unroll
              for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(t_o + q * 32, o);
                tmem_wait_ld();
                tmem_fix(o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                tmem_st32(t_o + q * 32, o);
              }
            }
            // the first part of P (and a rescaled O) is in TMEM: its PV MMAs may start
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_half[t]);
          }
        }
        const float2 s01 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        l = l * f + (s01.x + s01.y);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[t]);
      }
      sb += static_cast<uint32_t>(cnt);

      if (D == 128 && !wk.split) {
        // Two-tile unit: the epilogue warpgroup normalises and stores O_t. Hand
        // it 1/l of this group's rows (once it has read the previous unit's),
        // write the LSE here and go on to the next unit.
        const int q_local = r.q_local0 + t * BM + row;
        if (ok && p.lse != nullptr && q_local < r.lq)
          p.lse[static_cast<int64_t>(head) * p.lse_ld + r.q_row0 + q_local] = (m + __log2f(l)) * 0.69314718055994531f;
        if (ok && nwg > 0) ok = __all_sync(0xffffffffu, wait_bounded(&bars->il_free[t], (nwg - 1) & 1u, wc, 17));
        (t == 0 ? bars->xm : bars->xl)[row] = 1.f / l;
        mbar_arrive(&bars->il_full[t]);
        ++nwg;
        od0 += 1u;
        od1 += 1u;
        ++uk;
        continue;
      }

      // ---- epilogue: normalise and store (in split mode group 0 merges both halves)
      const int q_local = r.q_local0 + (wk.split ? 0 : t) * BM + row;
      const bool live = q_local < r.lq;
      const int64_t out_row = static_cast<int64_t>(r.q_row0) + q_local;
      const bool merge = wk.split && wk.count(1) > 0;
      const uint32_t w0 = od0, w1 = od1;   // this unit's o_done phases
      od0 += 1u;
      od1 += (!wk.split || wk.count(1) > 0) ? 1u : 0u;
      if (wk.split && t == 1) {
        // hand (m, l) to group 0, then wait until it has read them and O_1:
        // this group's next P (and so the next PV into O_1) comes only after.
        // xm / xl last carried 1/l to the epilogue warpgroup, which must be
        // done with every two-tile unit so far (four warps count each).
        if (D == 128 && ok && nwg > nwg_seen) {
          ok = __all_sync(0xffffffffu, wait_count(&bars->stage_done, static_cast<int>(4 * nwg), wc, 18));
          nwg_seen = nwg;
        }
        bars->xm[row] = (ok && cnt > 0) ? m : -INFINITY;
        bars->xl[row] = (ok && cnt > 0) ? l : 0.f;
        mbar_arrive(&bars->x_full);
        if (ok) ok = __all_sync(0xffffffffu, wait_bounded(&bars->x_empty, nx & 1u, wc, 9));
        ++nx;
        ++uk;
        continue;
      }
      if (wk.split && ok) ok = __all_sync(0xffffffffu, wait_bounded(&bars->x_full, nx & 1u, wc, 9));
      if (ok) {
        ok = wait_bounded(&bars->o_done[t], (t == 0 ? w0 : w1) & 1u, wc, 6);
        if (ok && merge) ok = wait_bounded(&bars->o_done[1], w1 & 1u, wc, 6);
        ok = __all_sync(0xffffffffu, ok);
      }
      // one part of a key-split last block publishes fp32 rows and their log2-sum-exp
      float* pdst = parts > 1 ? S.ws_part + ((static_cast<int64_t>(head) * kMaxTailSplit + part) * BM + row) * (D + 4)
                              : nullptr;
      if (ok) {
        tc_fence_after();
        float f0 = 1.f, f1 = 0.f;
        if (merge) {
          const float m1 = bars->xm[row], l1 = bars->xl[row];
          const float mm = fmaxf(m, m1);
          f0 = ex2_approx(m - mm);
          f1 = ex2_approx(m1 - mm);
          l = l * f0 + l1 * f1;
          m = mm;
        }
        const float inv_l = 1.f / l;
        f0 *= inv_l;
        f1 *= inv_l;
        __nv_bfloat16* dst = p.o + (out_row * p.n_heads + head) * D;
        const uint32_t t_o1 = tmem + lane_base + 256 + 128;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
          tmem_wait_ld();
          tmem_fix(o);
          if (merge) {
            uint32_t o1[32];
            tmem_ld32(t_o1 + c * 32, o1);
            tmem_wait_ld();
            tmem_fix(o1);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * f0 + __uint_as_float(o1[i]) * f1);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f0);
          }
          if (live) {
            if (pdst) {
              float4* d4 = reinterpret_cast<float4*>(pdst + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                    __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
            } else {
              uint4 pkt[4];
              uint32_t* w = reinterpret_cast<uint32_t*>(pkt);
#pragma unroll
              for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
              uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i) d4[i] = pkt[i];
            }
          }
        }
        if (live) {
          const float lse2 = m + __log2f(l);
          if (pdst)
            pdst[D] = lse2;
          else if (p.lse != nullptr)
            p.lse[static_cast<int64_t>(head) * p.lse_ld + out_row] = lse2 * 0.69314718055994531f;
        }
      }
      // group 1 may go on: its (m, l) and O_1 have been read
      if (wk.split) {
        tc_fence_before();
        mbar_arrive(&bars->x_empty);
        ++nx;
      }
      if (parts > 1) {
        // Every part has published its rows; the last part to arrive merges them.
        // The counter holds (epoch << 4 | arrivals): raising it to this call's
        // epoch first discards any count left by an earlier, aborted call. The
        // last part clears it once every part has arrived, so that a replay of
        // the same launch (a CUDA graph repeats the epoch) starts from zero.
        __threadfence();
        mbar_arrive(&bars->part_done);
        if (threadIdx.x == 0) {
          int last = 0;
          if (ok && wait_bounded(&bars->part_done, nk & 1u, wc, 10)) {
            int* ctr = S.ws_ctr + head;
            atomicMax(ctr, S.epoch << 4);
            const int old = atomicAdd(ctr, 1);
            last = ((old >> 4) == S.epoch) && ((old & 15) == parts - 1);
            if (last) atomicExch(ctr, 0);
          }
          bars->last = last;
          mbar_arrive(&bars->part_last);
        }
        if (ok) ok = __all_sync(0xffffffffu, wait_bounded(&bars->part_last, nk & 1u, wc, 10));
        ++nk;
        if (ok && bars->last)
          merge_key_parts<D>(S.ws_part + static_cast<int64_t>(head) * kMaxTailSplit * BM * (D + 4), parts,
                             min(BM, S.lq - r.q_local0), p.o, p.n_heads, head,
                             static_cast<int64_t>(S.q_row0) + r.q_local0, p.lse, p.lse_ld, warp % 4, lane);
      }
      ++uk;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The softmax warpgroups' setmaxnreg.inc can only be granted if the kernel is
// launched with the registers the split assumes; refuse to launch otherwise
// (an increase that cannot be granted would never return).
template <int D, int NSESS>
cudaError_t set_attr() {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, attn_kernel<D, NSESS>);
  if (e != cudaSuccess) return e;
  if (a.numRegs != kLaunchRegs || a.maxThreadsPerBlock < kAttnThreads) return cudaErrorInvalidConfiguration;
  return cudaFuncSetAttribute(attn_kernel<D, NSESS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<D>::kSmemBytes);
}

}  // namespace

int attn_smem_bytes(int head_dim) { return head_dim == 128 ? Cfg<128>::kSmemBytes : Cfg<64>::kSmemBytes; }

cudaError_t attn_prepare(int head_dim, int nsess_template) {
  if (head_dim == 128) return nsess_template == 1 ? set_attr<128, 1>() : set_attr<128, kAttnMaxBatch>();
  return nsess_template == 1 ? set_attr<64, 1>() : set_attr<64, kAttnMaxBatch>();
}

namespace {
template <int NSESS>
unsigned attn_grid(const AttnParams<NSESS>& p) {
  const int n = p.n_units;
  return static_cast<unsigned>(p.unit_ctr != nullptr ? std::min(n, sm_count()) : n);
}
}  // namespace

cudaError_t launch_attention_1(const AttnParams<1>& p, int head_dim, cudaStream_t st) {
  if (p.n_units <= 0) return cudaSuccess;
  if (head_dim == 128)
    return launch_dependent(attn_kernel<128, 1>, attn_grid(p), kAttnThreads, Cfg<128>::kSmemBytes, st, p);
  return launch_dependent(attn_kernel<64, 1>, attn_grid(p), kAttnThreads, Cfg<64>::kSmemBytes, st, p);
}

cudaError_t launch_attention_n(const AttnParams<kAttnMaxBatch>& p, int head_dim, cudaStream_t st) {
  if (p.n_units <= 0) return cudaSuccess;
  if (head_dim == 128)
    return launch_dependent(attn_kernel<128, kAttnMaxBatch>, attn_grid(p), kAttnThreads, Cfg<128>::kSmemBytes, st,
                            p);
  return launch_dependent(attn_kernel<64, kAttnMaxBatch>, attn_grid(p), kAttnThreads, Cfg<64>::kSmemBytes, st, p);
}

// ---------------------------------------------------------------- diagnostics
namespace {
// Waits on a barrier that nothing ever completes, with the same bounded wait
// the attention kernel uses, so that the time-out path can be exercised
// without any copy or tensor-core operation in flight.
__global__ void debug_wait_kernel(int32_t* err_word, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  WaitCtx wc{&abort_flag, err_word, timeout_ns};
  if (threadIdx.x == 0) (void)wait_bounded(&bar, 0, wc, 0xFF);
}
}  // namespace

cudaError_t launch_debug_wait(int32_t* err_word, uint64_t timeout_ns, cudaStream_t st) {
  return launch_plain(debug_wait_kernel, 1, 32, st, err_word, timeout_ns);
}

}  // namespace sr
