// kv_slot_mapping.cu -- token -> cache slot, through a block table ("paged")
// or through contiguous range descriptors ("range").
//
// Sources: "Blocktabelle", Datenfluss (the slot-mapping kernel: block index
// pos // block_size, table lookup, slot = block * block_size + offset, tail
// padded with PAD); "Range-addressed KV cache blocks ...", The Innovation
// (physical_block = range_start + (pos // block_size - range_cum), descriptor
// loaded once per position block, positions outside every range padded).
//
// GPU shape.  The pages' kernel runs one program per request and walks its
// tokens, which leaves a 128K-token request on one SM.  Here a CTA owns a
// fixed tile of 256 x TPT consecutive tokens (TPT per thread, coalesced, all
// of a thread's loads in flight together), so the grid depends only on
// max_num_tokens (stable under CUDA-graph capture) and long prefills spread
// over every SM.  TPT is 1 for batches up to a few hundred thousand tokens
// (the shortest dependency chain per thread, measured 1.2-6 us faster on
// decode and mixed batches than 4), then 4 (paged) or 4-8 (range); the
// thresholds were measured per map (see the *_tokens_per_thread rules).
// Each thread finds its request by a binary search of query_start_loc staged
// in shared memory.  The tail [num_tokens, max_num_tokens) is just more tiles
// that store PAD.
#include "kv_slot_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;

// Context-parallel filter: a table entry names a virtual block of T * W
// tokens dealt to the W ranks in chunks of I tokens, round robin; this rank
// keeps its own tokens (element ((p % (T*W)) / (I*W)) * I + p % I of its
// physical block) and pads the others.  W = 1 is the plain paged map.
struct CpArgs {
  int32_t world, rank;
  BlockDiv chunk;   // I
  BlockDiv ranks;   // W
  BlockDiv virt;    // T * W
  BlockDiv stripe;  // I * W
};

// Index arithmetic of the paged kernel: 64-bit in general, 32-bit when the
// host has checked that table offsets, in-row positions and slots all fit
// int32 (positions are 64-bit, so one 64-bit compare guards the narrowing),
// or the context-parallel filter.
enum class PagedMode { kWide, kNarrow, kCP };

template <int kTokPerThread, PagedMode kMode>
__global__ void __launch_bounds__(kThreads)
slot_mapping_paged_kernel(SlotArgs a, const int32_t* __restrict__ table, int32_t stride,
                          bool qsl_in_smem, CpArgs cp) {
  constexpr bool kCP = kMode == PagedMode::kCP;
  pdl_allow_next();
  pdl_wait();
  extern __shared__ int32_t s_qsl[];
  const int32_t base = blockIdx.x * (kThreads * kTokPerThread) + threadIdx.x;
  // positions do not depend on the request: start their loads first
  int64_t p[kTokPerThread];
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    p[k] = t < a.num_tokens ? a.positions[t] : 0;
  }
  uint32_t err = 0;
  const int32_t* q = stage_qsl(a, s_qsl, qsl_in_smem);
  check_qsl(a, q, err);  // in the shadow of the position loads
  // phase 1: table index of every token of the thread (-1: PAD without lookup)
  int64_t idx[kTokPerThread], off[kTokPerThread];
  int last_r = -1;
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    idx[k] = -1;
    off[k] = 0;
    if (t < a.num_tokens) {
      const int r = kTokPerThread == 1 ? request_of_guess(q, a.num_reqs, t)
                                       : request_of_cached(q, a.num_reqs, t, last_r);
      if (r >= 0) {
        if (p[k] < 0) {
          err |= KV_ERR_BAD_POSITION;
        } else if (kCP) {
          int64_t c, in_chunk, owner_q, owner, lb, v, stripe, unused;
          cp.chunk.divmod(p[k], c, in_chunk);
          cp.ranks.divmod(c, owner_q, owner);
          if (owner == cp.rank) {
            cp.virt.divmod(p[k], lb, v);
            cp.stripe.divmod(v, stripe, unused);
            off[k] = stripe * cp.chunk.size + in_chunk;
            if (lb < stride) idx[k] = (int64_t)r * stride + lb;
          }
        } else if (kMode == PagedMode::kNarrow) {
          // p < stride * T <= INT32_MAX: 32-bit block index and offset
          if (p[k] < (int64_t)stride * a.bs.size) {
            const uint32_t pu = (uint32_t)p[k];
            const uint32_t lb = a.bs.shift >= 0 ? pu >> a.bs.shift : pu / (uint32_t)a.bs.size;
            off[k] = (int32_t)(pu - lb * (uint32_t)a.bs.size);
            idx[k] = r * stride + (int32_t)lb;
          }
        } else {
          int64_t lb;
          a.bs.divmod(p[k], lb, off[k]);
          if (lb < stride) idx[k] = (int64_t)r * stride + lb;
        }
      }
    }
  }
  // phase 2: all table loads in flight together.  (Requesting the entry of
  // the decode guess "request t owns token t" before the search was measured
  // here: it waits on the position first, and came out 0.5 us slower.)
  int32_t blk[kTokPerThread];
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) blk[k] = idx[k] >= 0 ? table[idx[k]] : kNull;
  // phase 3: slots
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    if (t >= a.max_num_tokens) continue;
    if (kMode == PagedMode::kNarrow) {
      // num_blocks * T <= INT32_MAX: the slot of a valid block fits int32
      const int32_t b = blk[k];
      int64_t slot = kPad;
      if (b != kNull) {
        if (b < 0 || b >= a.num_blocks) err |= KV_ERR_BAD_BLOCK;
        else slot = b * a.bs.size + (int32_t)off[k];
      }
      a.slot_mapping[t] = slot;
    } else {
      a.slot_mapping[t] = slot_of(blk[k], off[k], a.bs.size, a.num_blocks, err);
    }
  }
  report(a.err, err);
}

// ---------------------------------------------------------------------------
// Range variant.  For a warp whose 32 tokens belong to one request (prefill,
// long context) the request's descriptors are read 32 at a time, one per
// lane; a warp scan turns the lengths into range ends, and each lane finds
// its range with a 5-step binary search over the lanes (shuffles).  The loop
// stops as soon as every lane is resolved, so the steady state of one range
// per request costs one descriptor load per 32 positions.  Warps that mix
// requests (decode batches) let each lane walk its own request's few ranges.
// Rows with a bad count or bad lengths are flagged by a separate grid-wide
// sweep over every request, so the error word does not depend on which
// descriptors the token loop happened to read.

// Warp path: all needing lanes share request r0.  Chunk 0 (descriptors
// 0..31, one per lane) arrives already scanned: `end0` is the end of lane's
// range, `s0`/`len0` its start and length, `total0` the chunk's total.  The
// warp keeps chunk 0 across its token groups, so a request with at most 32
// ranges costs one descriptor load per warp for all of the warp's tokens.
// A resolved range as a window of logical blocks [lo, hi) starting at block start.
struct RangeWindow {
  int r = -1;
  int64_t lo = 0, hi = 0, start = 0;
  __device__ __forceinline__ bool has(int rr, int64_t lb) const {
    return rr == r && lb >= lo && lb < hi;
  }
};

__device__ __forceinline__ void range_search_chunk(int64_t end, int32_t s, int32_t len,
                                                   int64_t cum_base, int64_t total, bool need,
                                                   int64_t lb, RangeWindow& win, bool& found) {
  // first lane j whose range ends past lb
  int lo = 0, hi = 31;
#pragma unroll
  for (int it = 0; it < 5; ++it) {
    const int mid = (lo + hi) >> 1;
    const int64_t v = __shfl_sync(kFull, end, mid);
    if (lo < hi) {
      if (v > lb) hi = mid; else lo = mid + 1;
    }
  }
  const int32_t sj = __shfl_sync(kFull, s, lo);
  const int64_t endj = __shfl_sync(kFull, end, lo);
  const int32_t lenj = __shfl_sync(kFull, len, lo);
  if (need && !found && lb >= cum_base && lb < cum_base + total) {
    found = true;
    win.lo = endj - lenj;
    win.hi = endj;
    win.start = sj;
  }
}

__device__ __forceinline__ void range_lookup_warp(const int32_t* __restrict__ rs,
                                                  const int32_t* __restrict__ rl, int nr,
                                                  int64_t end0, int32_t s0, int32_t len0,
                                                  int64_t total0, bool need, int64_t lb,
                                                  RangeWindow& win, bool& found) {
  const int lane = threadIdx.x & 31;
  range_search_chunk(end0, s0, len0, 0, total0, need, lb, win, found);
  int64_t cum_base = total0;
  for (int c0 = 32; c0 < nr && __any_sync(kFull, need && !found); c0 += 32) {
    const int i = c0 + lane;
    int32_t s = 0, len = 0;
    if (i < nr) {
      s = rs[i];
      len = max(rl[i], 0);
    }
    const int64_t incl = warp_inclusive_scan<int64_t>((int64_t)len);
    const int64_t total = __shfl_sync(kFull, incl, 31);
    range_search_chunk(cum_base + incl, s, len, cum_base, total, need, lb, win, found);
    cum_base += total;
  }
}

constexpr int kLanePrefetch = 4;  // descriptors a lane requests with the count (one int4)

// The first kLanePrefetch descriptors of one row (`rs`, `rl` point at the
// row): one 16-byte load each for starts and lengths when rows are 16-byte
// aligned, else four scattered loads.
__device__ __forceinline__ void lane_prefetch(const int32_t* __restrict__ rs,
                                              const int32_t* __restrict__ rl, int32_t rstride,
                                              bool vec4, int32_t (&pre_s)[kLanePrefetch],
                                              int32_t (&pre_l)[kLanePrefetch]) {
  if (vec4) {
    const int4 s4 = *reinterpret_cast<const int4*>(rs);
    const int4 l4 = *reinterpret_cast<const int4*>(rl);
    pre_s[0] = s4.x;
    pre_s[1] = s4.y;
    pre_s[2] = s4.z;
    pre_s[3] = s4.w;
    pre_l[0] = l4.x;
    pre_l[1] = l4.y;
    pre_l[2] = l4.z;
    pre_l[3] = l4.w;
  } else {
#pragma unroll
    for (int i = 0; i < kLanePrefetch; ++i) {
      pre_s[i] = i < rstride ? rs[i] : 0;
      pre_l[i] = i < rstride ? rl[i] : 0;
    }
  }
}

template <int kTokPerThread>
__global__ void __launch_bounds__(kThreads)
slot_mapping_range_kernel(SlotArgs a, const int32_t* __restrict__ range_start,
                          const int32_t* __restrict__ range_len,
                          const int32_t* __restrict__ num_ranges, int32_t rstride,
                          bool qsl_in_smem, bool vec4) {
  pdl_allow_next();
  pdl_wait();
  extern __shared__ int32_t s_qsl[];
  // positions staged per thread in shared memory: all loads are issued at
  // once, and the token loop below stays rolled (one copy of its search
  // paths keeps the instruction footprint small)
  __shared__ int64_t s_pos[kTokPerThread][kThreads];
  const int32_t base = blockIdx.x * (kThreads * kTokPerThread) + threadIdx.x;
  const int lane = threadIdx.x & 31;
  // the position loads and the qsl staging loads are in flight together; the
  // positions reach shared memory only after the staging barrier
  int64_t p[kTokPerThread];
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    p[k] = t < a.num_tokens ? a.positions[t] : 0;
  }
  // One token per thread (batches that fit one wave): a decode batch gives
  // request t its token t, so request t's first descriptors and count are
  // requested now, with the position, and used when the search confirms the
  // guess (a wrong guess only costs the unused loads; measured -0.8 us at
  // decode).
  constexpr bool kGuess = kTokPerThread == 1;
  int32_t g_s[kLanePrefetch] = {}, g_l[kLanePrefetch] = {}, g_nr = 0;
  bool g_ok = false;
  if constexpr (kGuess) {
    if (base < a.num_tokens && base < a.num_reqs && rstride > 0) {
      lane_prefetch(range_start + (int64_t)base * rstride, range_len + (int64_t)base * rstride,
                    rstride, vec4, g_s, g_l);
      g_nr = num_ranges[base];
      g_ok = true;
    }
  }
  uint32_t err = 0;
  const int32_t* q = stage_qsl(a, s_qsl, qsl_in_smem);
  check_qsl(a, q, err);  // in the shadow of the position loads
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) s_pos[k][threadIdx.x] = p[k];
  // the warp's scanned chunk 0 of request c_r (c_nr < 0: malformed row)
  int c_r = -1, c_nr = -1;
  int32_t c_s = 0, c_len = 0;
  int64_t c_end = 0, c_total = 0;

  // descriptor-row validation, every request, grid-wide: the thread's first
  // row is requested now and checked after the token loop, so the check costs
  // no round trip on the loop's critical path
  RangeRowCheck first_row;
  {
    unsigned r0, step;
    if (grid_first(a.num_reqs, r0, step))
      first_row.load(num_ranges, range_len, (int)r0, rstride, vec4);
  }

  RangeWindow win;  // this lane's last resolved range
  ReqSpan last_r;
#pragma unroll 1
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    const int64_t pk = s_pos[k][threadIdx.x];
    // every lane of the warp reaches the votes and shuffles below: no early exit
    const int r = t >= a.num_tokens   ? -1
                  : kTokPerThread == 1 ? request_of_guess(q, a.num_reqs, t)
                                       : request_of_cached(q, a.num_reqs, t, last_r);
    bool need = false;
    if (r >= 0) {
      if (pk < 0) err |= KV_ERR_BAD_POSITION;
      else need = true;
    }
    int64_t lb = 0, off = 0;
    if (need) a.bs.divmod(pk, lb, off);
    // arithmetic only while the position stays inside the lane's last range
    bool found = need && win.has(r, lb);
    const bool miss = need && !found;
    const unsigned missers = __ballot_sync(kFull, miss);
    if (missers != 0u) {
      const int r0 = __shfl_sync(kFull, r, __ffs(missers) - 1);
      if (__all_sync(kFull, !miss || r == r0)) {
        const int32_t* rs0 = range_start + (int64_t)r0 * rstride;
        const int32_t* rl0 = range_len + (int64_t)r0 * rstride;
        if (r0 != c_r) {
          // descriptor `lane` is requested together with the count
          int32_t pre_s = 0, pre_l = 0;
          if (lane < rstride) {
            pre_s = rs0[lane];
            pre_l = rl0[lane];
          }
          const int nr0 = num_ranges[r0];
          c_r = r0;
          c_nr = (nr0 >= 0 && nr0 <= rstride) ? nr0 : -1;  // malformed: PAD (the sweep flags it)
          c_s = lane < c_nr ? pre_s : 0;
          c_len = lane < c_nr ? max(pre_l, 0) : 0;
          c_end = warp_inclusive_scan<int64_t>((int64_t)c_len);
          c_total = __shfl_sync(kFull, c_end, 31);
        }
        if (c_nr >= 0) {
          bool got = false;
          range_lookup_warp(rs0, rl0, c_nr, c_end, c_s, c_len, c_total, miss, lb, win, got);
          if (got) {
            win.r = r;
            found = true;
          }
        }
      } else if (miss) {
        const int32_t* rs = range_start + (int64_t)r * rstride;
        const int32_t* rl = range_len + (int64_t)r * rstride;
        int32_t pre_s[kLanePrefetch], pre_l[kLanePrefetch];
        int nr;
        if (kGuess && g_ok && r == base) {
#pragma unroll
          for (int i = 0; i < kLanePrefetch; ++i) {
            pre_s[i] = g_s[i];
            pre_l[i] = g_l[i];
          }
          nr = g_nr;
        } else {
          lane_prefetch(rs, rl, rstride, vec4, pre_s, pre_l);
          nr = num_ranges[r];
        }
        if (nr >= 0 && nr <= rstride) {
          int64_t cum = 0;
#pragma unroll
          for (int i = 0; i < kLanePrefetch; ++i) {
            if (!found && i < nr) {
              const int64_t len = max(pre_l[i], 0);
              if (lb < cum + len) {
                win.r = r;
                win.lo = cum;
                win.hi = cum + len;
                win.start = pre_s[i];
                found = true;
              }
              cum += len;
            }
          }
          for (int i = kLanePrefetch; !found && i < nr; ++i) {
            const int64_t len = max(rl[i], 0);
            if (lb < cum + len) {
              win.r = r;
              win.lo = cum;
              win.hi = cum + len;
              win.start = rs[i];
              found = true;
            }
            cum += len;
          }
        }
      }
    }
    if (t < a.max_num_tokens)
      a.slot_mapping[t] =
          found ? slot_of(win.start + (lb - win.lo), off, a.bs.size, a.num_blocks, err) : kPad;
  }
  {
    unsigned r, step;  // this thread's rows: the first was loaded above
    if (grid_first(a.num_reqs, r, step)) {
      if (first_row.malformed(range_len, rstride)) err |= KV_ERR_BAD_RANGE;
      while (grid_next(a.num_reqs, r, step))
        if (range_row_malformed(num_ranges, range_len, (int)r, rstride)) err |= KV_ERR_BAD_RANGE;
    }
  }
  report(a.err, err);
}

// ---------------------------------------------------------------------------
// Range variant for large prefill batches and long contexts (4 or 8 tokens
// per thread, requests long enough to fill a tile).  A CTA whose token tile
// belongs to at most kStageReqs requests stages, for each of them, the count
// and the first kStageCap descriptors in shared memory: one warp per request,
// one load per descriptor, one warp scan turning the lengths into range ends
// (logical block ranges [end_{i-1}, end_i)).  A token resolves its block from
// there by a binary search for the first end past its logical block; when the
// whole tile lies in one request, a range whose blocks are all valid becomes
// a window of positions whose slot is the position plus a constant, so a
// token inside the range its thread resolved last costs one addition -- the
// descriptor once per position block, arithmetic per position.  Tiles of more
// requests, or a request of more than kStageCap ranges, let each thread walk
// its own request's ranges.  The grid-wide sweep over every descriptor row
// sets BAD_RANGE as in the kernel above.

constexpr int kStageReqs = 8;  // requests a CTA stages (one warp each)
constexpr int kStageCap = 32;  // descriptors staged per request (one per lane)
static_assert(kStageReqs == kThreads / 32, "one warp stages each request");

// Logical block lb of request r by a walk of its descriptor row in global
// memory (nr: its count), for tiles that could not be staged.  Sets win on
// success.
__device__ __forceinline__ bool range_walk(const int32_t* __restrict__ rs,
                                                 const int32_t* __restrict__ rl, int nr, int r,
                                                 int64_t lb, RangeWindow& win) {
  int64_t cum = 0;
  for (int i = 0; i < nr; ++i) {
    const int64_t len = max(rl[i], 0);
    if (lb < cum + len) {
      win = RangeWindow{r, cum, cum + len, rs[i]};
      return true;
    }
    cum += len;
  }
  return false;
}

// Staged row j (counts in s_cnt, range ends in s_end, starts in s_beg):
// the range holding logical block lb, or false when no range does.
__device__ __forceinline__ bool staged_find(const int64_t (*s_end)[kStageCap],
                                            const int32_t (*s_beg)[kStageCap],
                                            const int32_t* s_cnt, int j, int r, int64_t lb,
                                            RangeWindow& win) {
  const int n = s_cnt[j];
  const int64_t* e = s_end[j];
  if (n <= 0 || lb >= e[n - 1]) return false;
  int lo = 0, hi = n - 1;
  while (lo < hi) {  // first range whose end passes lb
    const int mid = (lo + hi) >> 1;
    if (e[mid] > lb) hi = mid; else lo = mid + 1;
  }
  win = RangeWindow{r, lo > 0 ? e[lo - 1] : 0, e[lo], s_beg[j][lo]};
  return true;
}

// Positions [plo, phi) of one range whose blocks are all valid: slot p + delta.
struct PosWindow {
  int64_t plo = 0, phi = 0, delta = 0;
  __device__ __forceinline__ bool has(int64_t p) const { return p >= plo && p < phi; }
};

// Slot of position p of request r (the staged row 0) when p is outside the
// position window: resolve its range, and make that range the window when
// all its blocks are valid.
__device__ __forceinline__ int64_t window_miss(int64_t p, const SlotArgs& a,
                                               const int64_t (*s_end)[kStageCap],
                                               const int32_t (*s_beg)[kStageCap],
                                               const int32_t* s_cnt, int r, RangeWindow& win,
                                               PosWindow& pw, uint32_t& err) {
  if (p < 0) {
    err |= KV_ERR_BAD_POSITION;
    return kPad;
  }
  const int64_t T = a.bs.size;
  int64_t lb, off;
  a.bs.divmod(p, lb, off);
  if (!win.has(r, lb) && !staged_find(s_end, s_beg, s_cnt, 0, r, lb, win)) return kPad;
  // block_size < 2^31, so ends below 2^32 keep hi * T inside int64
  if (win.start >= 1 && win.start + (win.hi - win.lo) <= a.num_blocks &&
      win.hi <= (INT64_MAX >> 31)) {
    pw.plo = win.lo * T;
    pw.phi = win.hi * T;
    pw.delta = (win.start - win.lo) * T;
  }
  return slot_of(win.start + (lb - win.lo), off, a.bs.size, a.num_blocks, err);
}

// At most 64 registers (it needs 56): four CTAs per SM keep the grid within
// one wave (512 CTAs for 1M positions at 8 tokens per thread); an earlier
// form at 80 registers ran three per SM and needed a second wave.
template <int kTokPerThread>
__global__ void __launch_bounds__(kThreads, 4)
slot_mapping_range_staged_kernel(SlotArgs a, const int32_t* __restrict__ range_start,
                                 const int32_t* __restrict__ range_len,
                                 const int32_t* __restrict__ num_ranges, int32_t rstride,
                                 bool qsl_in_smem, bool vec4) {
  pdl_allow_next();
  pdl_wait();
  extern __shared__ int32_t s_qsl[];
  __shared__ int64_t s_end[kStageReqs][kStageCap];  // staged range ends
  __shared__ int32_t s_beg[kStageReqs][kStageCap];  // staged range starts
  // positions staged per thread in shared memory: the token loops stay
  // rolled (one copy of their search paths keeps the instruction footprint
  // small) and no register holds a position while it is in flight; only the
  // thread itself reads its entries back
  __shared__ int64_t s_pos[kTokPerThread][kThreads];
  __shared__ int32_t s_cnt[kStageReqs];  // staged counts, -1: malformed row
  constexpr int32_t kTile = kThreads * kTokPerThread;
  const int32_t t_lo = blockIdx.x * kTile;
  const int32_t base = t_lo + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  // the positions go straight to shared memory by asynchronous copies, in
  // flight together with the qsl and descriptor staging loads below
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    if (t < a.num_tokens) cp_async8(&s_pos[k][threadIdx.x], a.positions + t);
    else s_pos[k][threadIdx.x] = 0;
  }
  uint32_t err = 0;
  const int32_t* q = stage_qsl(a, s_qsl, qsl_in_smem);
  check_qsl(a, q, err);  // in the shadow of the position loads

  // descriptor-row validation, every request, grid-wide: the thread's first
  // row is requested now and checked after the token loop, so the check costs
  // no round trip on the loop's critical path
  RangeRowCheck first_row;
  {
    unsigned r0, step;
    if (grid_first(a.num_reqs, r0, step))
      first_row.load(num_ranges, range_len, (int)r0, rstride, vec4);
  }

  // Requests of this tile: [st_lo, st_lo + st_n) when at most kStageReqs
  // (every thread computes the same, CTA-uniform values).
  const int32_t t_hi = min(t_lo + kTile, a.num_tokens);
  int st_lo = 0, st_n = 0;
  if (t_lo < t_hi && a.num_reqs > 0) {
    const int r0 = max(find_span(q, a.num_reqs, t_lo), 0);
    const int r1 = find_span(q, a.num_reqs, t_hi - 1);
    if (r1 >= r0 && r1 - r0 < kStageReqs) {
      st_lo = r0;
      st_n = r1 - r0 + 1;
    }
  }
  if (st_n > 0) {
    // warp j stages row st_lo + j: the count and the first kStageCap
    // descriptors (one per lane) in one round trip, the lengths scanned into
    // range ends (lengths <= 0 count as empty; a malformed count -1, all PAD)
    if (wid < st_n) {
      const int r = st_lo + wid;
      const int raw = num_ranges[r];
      int32_t st = 0, ln = 0;
      if (lane < rstride) {
        st = range_start[(int64_t)r * rstride + lane];
        ln = range_len[(int64_t)r * rstride + lane];
      }
      const int n = (raw >= 0 && raw <= rstride) ? raw : -1;
      const int64_t end = warp_inclusive_scan<int64_t>(lane < n ? (int64_t)max(ln, 0) : 0);
      s_end[wid][lane] = end;
      s_beg[wid][lane] = st;
      if (lane == 0) s_cnt[wid] = n;
    }
    __syncthreads();
    // a row of more than kStageCap ranges does not fit: the whole CTA takes
    // the general path (the same decision in every thread)
    for (int j = 0; j < st_n; ++j)
      if (s_cnt[j] > kStageCap) st_n = 0;
  }

  const int32_t T = a.bs.size;
  cp_async_wait_all();  // this thread's positions are in s_pos
  if (st_n == 1 && q[st_lo] <= t_lo && t_hi <= q[st_lo + 1]) {
    // Every token of the tile belongs to request st_lo.  A resolved range
    // whose blocks all lie in [1, num_blocks) becomes a window of positions
    // [plo, phi) whose slot is p + delta: no division, no lookup.
    PosWindow pw;
    RangeWindow win;
    int64_t* out = a.slot_mapping + base;
    if (t_lo + kTile <= a.num_tokens) {
      // a full tile: every token is valid and below max_num_tokens
#pragma unroll 1
      for (int k = 0; k < kTokPerThread; ++k, out += kThreads) {
        const int64_t pk = s_pos[k][threadIdx.x];
        *out = pw.has(pk) ? pk + pw.delta
                          : window_miss(pk, a, s_end, s_beg, s_cnt, st_lo, win, pw, err);
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < kTokPerThread; ++k, out += kThreads) {
        const int32_t t = base + k * kThreads;
        if (t >= a.max_num_tokens) break;
        int64_t slot = kPad;
        if (t < a.num_tokens) {
          const int64_t pk = s_pos[k][threadIdx.x];
          slot = pw.has(pk) ? pk + pw.delta
                            : window_miss(pk, a, s_end, s_beg, s_cnt, st_lo, win, pw, err);
        }
        *out = slot;
      }
    }
  } else {
    RangeWindow win;  // this thread's last resolved range
    ReqSpan last_r;
#pragma unroll 1
    for (int k = 0; k < kTokPerThread; ++k) {
      const int32_t t = base + k * kThreads;
      if (t >= a.max_num_tokens) break;
      const int64_t pk = s_pos[k][threadIdx.x];
      const int r = t < a.num_tokens ? request_of_cached(q, a.num_reqs, t, last_r) : -1;
      int64_t slot = kPad;
      if (r >= 0) {
        if (pk < 0) {
          err |= KV_ERR_BAD_POSITION;
        } else {
          int64_t lb, off;
          a.bs.divmod(pk, lb, off);
          bool found = win.has(r, lb);
          const int j = r - st_lo;
          if (!found && j >= 0 && j < st_n) {
            found = staged_find(s_end, s_beg, s_cnt, j, r, lb, win);
          } else if (!found) {
            const int32_t* rs = range_start + (int64_t)r * rstride;
            const int32_t* rl = range_len + (int64_t)r * rstride;
            const int nr = num_ranges[r];
            if (nr >= 0 && nr <= rstride) found = range_walk(rs, rl, nr, r, lb, win);
          }
          if (found) slot = slot_of(win.start + (lb - win.lo), off, T, a.num_blocks, err);
        }
      }
      a.slot_mapping[t] = slot;
    }
  }
  {
    unsigned r, step;  // this thread's rows: the first was loaded above
    if (grid_first(a.num_reqs, r, step)) {
      if (first_row.malformed(range_len, rstride)) err |= KV_ERR_BAD_RANGE;
      while (grid_next(a.num_reqs, r, step))
        if (range_row_malformed(num_ranges, range_len, (int)r, rstride)) err |= KV_ERR_BAD_RANGE;
    }
  }
  report(a.err, err);
}

// Tokens per thread, measured per map (ncu, cold caches, 262K-2.6M
// positions).  A wave is 4 resident CTAs per SM.
// Paged map: 1 while the grid is at most two waves (~311K tokens), else 4
// (4 beat 8 and 16 at every size: 7.1 vs 7.5 / 9.1 us at 1M positions,
// 11.6 vs 13.5 / 18.8 us at 2.6M).
int paged_tokens_per_thread(int32_t max_num_tokens) {
  const int64_t wave = (int64_t)sm_count() * 4;
  return ((int64_t)max_num_tokens + kThreads - 1) / kThreads <= 2 * wave ? 1 : 4;
}

// Range map: 1 while the grid fits one wave, else the smaller of 4 and 8
// that keeps the grid within about one wave (its per-token state is larger,
// and at 1M-2.6M positions 8 was level with or ahead of 4).
int range_tokens_per_thread(int32_t max_num_tokens) {
  const int64_t wave = (int64_t)sm_count() * 4;
  if (((int64_t)max_num_tokens + kThreads - 1) / kThreads <= wave) return 1;
  return ((int64_t)max_num_tokens + kThreads * 4 - 1) / (kThreads * 4) <= wave ? 4 : 8;
}

int grid_for(int32_t max_num_tokens, int tpt) {
  return max(1, (int)(((int64_t)max_num_tokens + kThreads * tpt - 1) / (kThreads * tpt)));
}

template <PagedMode kMode>
int launch_paged(const int32_t* query_start_loc, const int64_t* positions,
                 const int32_t* block_table, int32_t table_stride, int32_t num_reqs,
                 int32_t num_tokens, int32_t max_num_tokens, int32_t block_size,
                 int64_t num_blocks, int64_t* slot_mapping, int32_t* d_err, kv_stream_t stream,
                 const CpArgs& cp) {
  int rc = check_common(query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
                        block_size, num_blocks, slot_mapping);
  if (rc != KV_OK) return rc;
  if (table_stride < 0) return KV_EINVAL;
  if (num_reqs > 0 && num_tokens > 0 && table_stride > 0 &&
      (block_table == nullptr || !aligned(block_table, 4)))
    return KV_EINVAL;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if (max_num_tokens == 0 && num_reqs == 0) return KV_OK;
  const int tpt = paged_tokens_per_thread(max_num_tokens);
  const int grid = grid_for(max_num_tokens, tpt);
  const bool staged = num_reqs + 1 <= kQslSmemMax;
  const size_t smem = staged && num_reqs > 0 ? sizeof(int32_t) * (num_reqs + 1) : 0;
  SlotArgs a{query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
             BlockDiv::make(block_size), num_blocks, slot_mapping, d_err};
  const bool st = staged && num_reqs > 0;
  return launch_pdl(tpt == 1 ? slot_mapping_paged_kernel<1, kMode>
                              : slot_mapping_paged_kernel<4, kMode>,
                    grid, kThreads, smem, stream, a, block_table, table_stride, st, cp);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_slot_mapping_paged(const int32_t* query_start_loc, const int64_t* positions,
                                     const int32_t* block_table, int32_t table_stride,
                                     int32_t num_reqs, int32_t num_tokens,
                                     int32_t max_num_tokens, int32_t block_size,
                                     int64_t num_blocks, int64_t* slot_mapping, int32_t* d_err,
                                     kv_stream_t stream) {
  // 32-bit indices when every table offset, in-row position and slot fits int32
  const bool narrow = (int64_t)num_reqs * table_stride <= INT32_MAX &&
                      (int64_t)table_stride * block_size <= INT32_MAX &&
                      num_blocks * (int64_t)block_size <= INT32_MAX;
  if (narrow)
    return launch_paged<PagedMode::kNarrow>(query_start_loc, positions, block_table,
                                            table_stride, num_reqs, num_tokens, max_num_tokens,
                                            block_size, num_blocks, slot_mapping, d_err, stream,
                                            CpArgs{});
  return launch_paged<PagedMode::kWide>(query_start_loc, positions, block_table, table_stride,
                                        num_reqs, num_tokens, max_num_tokens, block_size,
                                        num_blocks, slot_mapping, d_err, stream, CpArgs{});
}

extern "C" int kv_slot_mapping_paged_cp(const int32_t* query_start_loc,
                                        const int64_t* positions, const int32_t* block_table,
                                        int32_t table_stride, int32_t num_reqs,
                                        int32_t num_tokens, int32_t max_num_tokens,
                                        int32_t block_size, int64_t num_blocks,
                                        int32_t cp_world_size, int32_t cp_rank,
                                        int32_t cp_interleave, int64_t* slot_mapping,
                                        int32_t* d_err, kv_stream_t stream) {
  if (cp_world_size < 1 || cp_rank < 0 || cp_rank >= cp_world_size || cp_interleave < 1 ||
      block_size <= 0)
    return KV_EINVAL;
  if (block_size % cp_interleave != 0) return KV_EUNSUPPORTED;
  if ((int64_t)block_size * cp_world_size > INT32_MAX ||
      (int64_t)cp_interleave * cp_world_size > INT32_MAX)
    return KV_EINVAL;
  const CpArgs cp{cp_world_size, cp_rank, BlockDiv::make(cp_interleave),
                  BlockDiv::make(cp_world_size), BlockDiv::make(block_size * cp_world_size),
                  BlockDiv::make(cp_interleave * cp_world_size)};
  return launch_paged<PagedMode::kCP>(query_start_loc, positions, block_table, table_stride,
                                      num_reqs,
                            num_tokens, max_num_tokens, block_size, num_blocks, slot_mapping,
                            d_err, stream, cp);
}

extern "C" int kv_slot_mapping_range(const int32_t* query_start_loc, const int64_t* positions,
                                     const int32_t* range_start, const int32_t* range_len,
                                     const int32_t* num_ranges, int32_t range_stride,
                                     int32_t num_reqs, int32_t num_tokens,
                                     int32_t max_num_tokens, int32_t block_size,
                                     int64_t num_blocks, int64_t* slot_mapping, int32_t* d_err,
                                     kv_stream_t stream) {
  int rc = check_common(query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
                        block_size, num_blocks, slot_mapping);
  if (rc != KV_OK) return rc;
  rc = check_ranges(range_start, range_len, num_ranges, range_stride, num_reqs);
  if (rc != KV_OK) return rc;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if (max_num_tokens == 0 && num_reqs == 0) return KV_OK;
  const int tpt = range_tokens_per_thread(max_num_tokens);
  const int grid = grid_for(max_num_tokens, tpt);
  const bool staged = num_reqs + 1 <= kQslSmemMax;
  const bool st = staged && num_reqs > 0;
  SlotArgs a{query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
             BlockDiv::make(block_size), num_blocks, slot_mapping, d_err};
  const bool v4 = rows_vec4(range_start, range_len, range_stride);
  const size_t qsl_smem = st ? sizeof(int32_t) * (num_reqs + 1) : 0;
  // Descriptor staging pays for large batches (beyond one wave of one token
  // per thread) whose tiles belong to few requests: on average at least
  // tile / kStageReqs / 2 tokens per request (prefill batches, long
  // contexts).  A decode or mixed batch keeps the kernel above (measured:
  // staging cost a mixed 8432-token batch 1 us, saved 1.7 us at 1M
  // positions).
  const int64_t tile = (int64_t)kThreads * tpt;
  if (tpt > 1 && range_stride > 0 && num_reqs > 0 &&
      (int64_t)num_tokens * kStageReqs * 2 >= tile * num_reqs) {
    const size_t smem = qsl_smem;
    const size_t static_smem = sizeof(int64_t) * tpt * kThreads +
                               (sizeof(int64_t) + sizeof(int32_t)) * kStageReqs * kStageCap +
                               sizeof(int32_t) * kStageReqs;
    auto kernel = tpt == 4 ? slot_mapping_range_staged_kernel<4>
                           : slot_mapping_range_staged_kernel<8>;
    if (smem + static_smem > 48 * 1024 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
      return KV_ECUDA;
    return launch_pdl(kernel, grid, kThreads, smem, stream, a, range_start, range_len,
                      num_ranges, range_stride, st, v4);
  }
  auto kernel = tpt == 1   ? slot_mapping_range_kernel<1>
                : tpt == 4 ? slot_mapping_range_kernel<4>
                           : slot_mapping_range_kernel<8>;
  return launch_pdl(kernel, grid, kThreads, qsl_smem, stream, a, range_start, range_len,
                    num_ranges, range_stride, st, v4);
}
