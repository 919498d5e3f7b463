// plan.cuh -- the split-KV partition shared by the attention kernels and the combine.
//
// Work is counted in key tiles of kTileKeys keys.  A query row that sees L keys
// owns ceil(L / kTileKeys) tiles; rows are laid out in order (request by request,
// query by query) to form one global tile sequence of length T.  Starting a row
// costs the pair several tiles' time (loading its Q, writing its output), so
// the sequence is split by cost: every non-empty row is preceded by kRowCost cost
// units, each tile is one unit, C = T + kRowCost * (non-empty rows), and worker w of G
// (a CTA pair) takes the tiles whose units fall in [floor(w*C/G), floor((w+1)*C/G)).
// A boundary that falls in a row's leading units gives the whole row to the next
// worker.  A row cut by a worker boundary is a split row: each worker that touches it
// writes a partial (normalised output + lse) and the worker holding the row's last
// tile owns the merge in the combine kernel, in worker order.
//
// This is the split-K partition of the Modular MAX "mla_decoding_single_batch"
// page (key range split across blocks, with exp-sum / max statistics merged
// afterwards) computed on the device from kv_indptr / qo_indptr, so that no host
// planning step (the FlashMLA get_mla_metadata step) is needed and the call can
// be captured in a CUDA graph.
#pragma once
#include <cstdint>

namespace mla {

constexpr int kTileKeys = 64;
constexpr int kRowCost = 5;  // cost units of starting a row (tuned on the benchmark batches over 2..8)

// Sum over x = 1..n of ceil(x / 64): the tiles of rows with lengths 1..n.
__device__ __forceinline__ long long cum_tiles(long long n) {
  if (n <= 0) return 0;
  long long a = n / kTileKeys, r = n % kTileKeys;
  return 32LL * a * (a + 1) + r * (a + 1);
}

__device__ __forceinline__ int row_tiles(long long len) {
  return len <= 0 ? 0 : (int)((len + kTileKeys - 1) / kTileKeys);
}

// Per-request geometry.  Decode is prefill with q_len = 1 and qo = b.
struct Req {
  int qo0;      // first query row of the request
  int q_len;    // query rows
  int kv0;      // first kv_indices entry of the request
  int kv_len;   // keys of the request
};

struct PlanArgs {
  const int32_t* kv_indptr;  // nullptr: every row owns `topk` consecutive entries
  const int32_t* qo_indptr;  // nullptr for decode
  int batch;
  int num_kv_indices;
  int topk;                  // entries per row when kv_indptr is nullptr (sparse decode)
};

__device__ __forceinline__ Req load_req(const PlanArgs& p, int b) {
  Req r;
  int k0, k1;
  if (p.kv_indptr) {
    k0 = __ldg(p.kv_indptr + b);
    k1 = __ldg(p.kv_indptr + b + 1);
  } else {  // sparse decode: row b lists its keys in entries b*topk .. b*topk + topk - 1
    k0 = b * p.topk;
    k1 = k0 + p.topk;
  }
  // Clamp so that corrupt indptr never leads to reads outside kv_indices.
  k0 = min(max(k0, 0), p.num_kv_indices);
  k1 = min(max(k1, k0), p.num_kv_indices);
  r.kv0 = k0;
  r.kv_len = k1 - k0;
  if (p.qo_indptr) {
    int q0 = __ldg(p.qo_indptr + b), q1 = __ldg(p.qo_indptr + b + 1);
    r.qo0 = q0;
    r.q_len = max(q1 - q0, 0);
  } else {
    r.qo0 = b;
    r.q_len = 1;
  }
  return r;
}

// Keys seen by query i of request r (bottom-right causal; decode: all keys).
__device__ __forceinline__ long long row_len(const Req& r, int i) {
  return (long long)r.kv_len - r.q_len + i + 1;
}

__device__ __forceinline__ long long req_tiles(const Req& r) {
  long long p = (long long)r.kv_len - r.q_len;
  return cum_tiles(p + r.q_len) - cum_tiles(p);
}

// Tiles owned by query rows 0..i-1 of request r.
__device__ __forceinline__ long long req_tiles_before(const Req& r, int i) {
  long long p = (long long)r.kv_len - r.q_len;
  return cum_tiles(p + i) - cum_tiles(p);
}

// Non-empty rows (rows that see at least one key) among query rows 0..i-1 of r; rows
// i < q_len - kv_len see no key.
__device__ __forceinline__ long long req_rows_before(const Req& r, int i) {
  return max(0LL, (long long)i - max(0LL, (long long)r.q_len - r.kv_len));
}

// Cost units of request r, and of its query rows 0..i-1.
__device__ __forceinline__ long long req_cost(const Req& r) {
  return req_tiles(r) + kRowCost * req_rows_before(r, r.q_len);
}
__device__ __forceinline__ long long req_cost_before(const Req& r, int i) {
  return req_tiles_before(r, i) + kRowCost * req_rows_before(r, i);
}

// Worker holding cost unit y (of C), and the first unit of worker w.
__device__ __forceinline__ int worker_of(long long y, long long C, int G) {
  return (int)(((y + 1) * (long long)G - 1) / C);
}

__device__ __forceinline__ long long worker_start(int w, long long C, int G) {
  return (long long)w * C / G;
}

// Where a worker starts: request, query row within it, tile within the row, and the
// global tile where it ends.
struct Cursor {
  int b;            // request
  int i;            // query row within the request
  int t;            // tile within the row
  long long g;      // global tile index
  long long tile0;  // global index of the request's first tile
  long long cost0;  // first cost unit of the request
  long long g_end;  // global tile index where the worker's range ends
};

// Executed by one full warp: the position of cost unit x (x < C) -- request b, query
// row i, tile t of the row, global tile g, and the request's first tile and cost unit.
// A unit in a row's leading kRowCost units maps to the row's first tile.
__device__ inline void warp_locate(const PlanArgs& p, long long x, Cursor* cur) {
  const int lane = threadIdx.x & 31;
  long long run_cost = 0, run_tiles = 0;
  for (int base = 0; base < p.batch; base += 32) {
    int b = base + lane;
    Req r;
    long long n = 0, nt = 0;
    if (b < p.batch) {
      r = load_req(p, b);
      nt = req_tiles(r);
      n = req_cost(r);
    }
    long long incl = n, incl_t = nt;
    for (int o = 1; o < 32; o <<= 1) {
      long long v = __shfl_up_sync(0xffffffffu, incl, o);
      long long vt = __shfl_up_sync(0xffffffffu, incl_t, o);
      if (lane >= o) {
        incl += v;
        incl_t += vt;
      }
    }
    const long long excl = run_cost + incl - n, excl_t = run_tiles + incl_t - nt;
    unsigned hit = __ballot_sync(0xffffffffu, n > 0 && excl <= x && x < excl + n);
    if (hit) {
      int src = __ffs(hit) - 1;
      if (lane == src) {
        // Largest query row i with cost_before(i) <= x - excl.
        const long long off = x - excl;
        int lo = 0, hi = r.q_len - 1;
        while (lo < hi) {
          int mid = (lo + hi + 1) >> 1;
          if (req_cost_before(r, mid) <= off) lo = mid; else hi = mid - 1;
        }
        const long long in_row = off - req_cost_before(r, lo) - kRowCost;
        cur->b = b;
        cur->i = lo;
        cur->t = (int)max(0LL, in_row);
        cur->tile0 = excl_t;
        cur->cost0 = excl;
        cur->g = excl_t + req_tiles_before(r, lo) + cur->t;
      }
      cur->b = __shfl_sync(0xffffffffu, cur->b, src);
      cur->i = __shfl_sync(0xffffffffu, cur->i, src);
      cur->t = __shfl_sync(0xffffffffu, cur->t, src);
      cur->tile0 = __shfl_sync(0xffffffffu, cur->tile0, src);
      cur->cost0 = __shfl_sync(0xffffffffu, cur->cost0, src);
      cur->g = __shfl_sync(0xffffffffu, cur->g, src);
      return;
    }
    run_cost += __shfl_sync(0xffffffffu, incl, 31);
    run_tiles += __shfl_sync(0xffffffffu, incl_t, 31);
  }
}

// Executed by one full warp.  Returns C (total cost units; 0 when there are no tiles)
// and the cursor at worker w's first tile, with the tile where its range ends.
__device__ inline long long warp_plan(const PlanArgs& p, int w, int G, Cursor* cur) {
  const int lane = threadIdx.x & 31;
  long long C = 0, T = 0;
  for (int base = 0; base < p.batch; base += 32) {
    int b = base + lane;
    long long n = 0, nt = 0;
    if (b < p.batch) {
      const Req r = load_req(p, b);
      nt = req_tiles(r);
      n = req_cost(r);
    }
    for (int o = 16; o > 0; o >>= 1) {
      n += __shfl_xor_sync(0xffffffffu, n, o);
      nt += __shfl_xor_sync(0xffffffffu, nt, o);
    }
    C += n;
    T += nt;
  }
  cur->b = p.batch;
  cur->i = 0;
  cur->t = 0;
  cur->g = T;
  cur->tile0 = T;
  cur->cost0 = C;
  cur->g_end = T;
  if (T == 0) return 0;
  const long long x0 = worker_start(w, C, G), x1 = worker_start(w + 1, C, G);
  if (x1 < C) {
    Cursor e;
    warp_locate(p, x1, &e);
    cur->g_end = e.g;
  }
  if (x0 < C) warp_locate(p, x0, cur);
  if (cur->g > cur->g_end) cur->g = cur->g_end;  // an empty range (all in leading units)
  return C;
}

// One segment of a worker's range: tiles [t_begin, t_end) of one query row.
struct Segment {
  int row;          // global query row (decode: request)
  int b;            // request
  int kv0;          // first kv_indices entry of the request
  int len;          // keys the row sees
  int t_begin, t_end;
  int slot;         // partial-result slot of this worker: 0 = first segment, 1 = other
  bool whole;       // the segment covers the whole row (final output written directly)
  bool first;       // first segment of this worker
  long long row_tile0;  // global index of the row's first tile
  long long row_cost0;  // first cost unit of the row (its leading kRowCost units)
};

// Sequential walk over a worker's segments (every thread of a CTA may run its own
// copy; all copies see the same sequence).
struct Walker {
  PlanArgs p;
  long long g, end;   // next global tile, end of the worker's range
  int b, i, t;
  long long req_tile0, req_cost0;
  Req r;
  bool started;

  __device__ void init(const PlanArgs& pa, const Cursor& c) {
    p = pa;
    g = c.g;
    end = c.g_end;
    b = c.b; i = c.i; t = c.t; req_tile0 = c.tile0; req_cost0 = c.cost0;
    started = false;
    if (g < end && b < p.batch) r = load_req(p, b);
  }

  __device__ bool next(Segment& s) {
    if (g >= end) return false;
    // Skip rows without tiles (empty requests, rows seeing no key).
    while (true) {
      if (i >= r.q_len) {
        req_tile0 += req_tiles(r);
        req_cost0 += req_cost(r);
        ++b;
        i = 0;
        t = 0;
        if (b >= p.batch) return false;
        r = load_req(p, b);
        continue;
      }
      if (row_tiles(row_len(r, i)) == 0) { ++i; t = 0; continue; }
      break;
    }
    const int nt = row_tiles(row_len(r, i));
    const long long avail = end - g;
    const int t_end = (int)min((long long)nt, (long long)t + avail);
    s.row = r.qo0 + i;
    s.b = b;
    s.kv0 = r.kv0;
    s.len = (int)row_len(r, i);
    s.t_begin = t;
    s.t_end = t_end;
    s.first = !started;
    s.slot = started ? 1 : 0;
    s.whole = (t == 0 && t_end == nt);
    s.row_tile0 = req_tile0 + req_tiles_before(r, i);
    s.row_cost0 = req_cost0 + req_cost_before(r, i);
    started = true;
    g += t_end - t;
    if (t_end == nt) { ++i; t = 0; } else { t = t_end; }
    return true;
  }
};

// Per-worker record read by the combine kernel.
struct CombineRecord {
  int row;         // row of this worker's first segment if that row is split; else -1
  int w_first;     // first worker holding a fragment of the row
  int slot_first;  // slot of that worker's fragment (every later worker holds it in slot 0)
  int w_last;      // last worker holding a fragment of the row (it owns the merge)
  int live;        // this worker has at least one tile (else it holds no fragment)
  int min_units;   // floor(C / G): >= kRowCost + 1 means no worker is empty
};

// Record for worker w given its first segment (or none): which split row the worker's
// slot-0 fragment belongs to, and the workers that share the row.
__device__ __forceinline__ CombineRecord make_record(bool has_first, const Segment& s, long long C, int G) {
  CombineRecord rec{-1, 0, 0, 0, has_first ? 1 : 0, C > 0 ? (int)min(C / G, 1LL << 30) : 0};
  if (has_first && !s.whole) {
    const long long y0 = s.row_cost0 + kRowCost;     // cost unit of the row's first tile
    const long long y1 = y0 + row_tiles(s.len) - 1;  // ... and of its last tile
    rec.row = s.row;
    rec.w_first = worker_of(y0, C, G);
    rec.w_last = worker_of(y1, C, G);
    // The row is w_first's first segment iff that worker's units start no earlier than
    // the row's leading units (else it holds tiles of earlier rows first).
    rec.slot_first = (worker_start(rec.w_first, C, G) >= s.row_cost0) ? 0 : 1;
  }
  return rec;
}

}  // namespace mla
