// mla_tc.cu -- paged MLA attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// one 2-CTA cluster per split-KV worker.
//
// What one worker computes: for each query row of its tile range (see plan.cuh) and
// all query heads at once (heads are the MMA M dimension, padded to 128):
//   S = Q . K^T over 64-key tiles, K = [ckv | kpe] gathered through kv_indices,
//   online softmax over S (running max, rescale, running sum: Modular MAX
//   "mla_decoding_single_batch", "Flash attention v2 algorithm"),
//   O += P . V with V = the ckv latent of the same tile (the same page says V is
//   K[:, :depth_v]; it is never loaded separately).
//
// How the pair splits the work.  O for 128 heads x 512 fp32 needs all 512 TMEM
// columns of an SM, which would leave none for S.  So CTA rank r owns
// O[:, 256r : 256r+256] and a 288-wide slice of the 576-wide query-key depth:
//   rank r: ckv[:, 256r : 256r+256] (its V columns too) and kpe[:, 32r : 32r+32].
// Each CTA computes a partial S over its depth slice; the two partial S tiles are
// swapped through distributed shared memory and added, so every score is computed
// once.  The partials travel as 24-bit floats (fp32 rounded to 16 significant bits,
// relative error <= 2^-16, 24 KB per 64-key tile instead of 32 KB).  Both CTAs add the
// same rounded values (fp32 addition commutes), so they see identical S and take
// identical softmax decisions.  This is the left/right split of the output that
// FlashMLA's "seesaw" schedule uses across two warpgroups (oL, oR), done here across
// the two SMs of a cluster with the depth split as well.
//
// The exchange is the pair's critical path: a one-way SM-to-SM transfer was measured at
// over a microsecond inside this kernel, about as long as a tile's HBM time.  Each
// softmax warp exchanges its own 3 KB piece (32 heads x 32 keys) with the warp of the
// same index in the peer, by st.async stores straight from registers that complete
// bytes on the peer warp's mbarrier, so no warp waits for another and nothing is staged.
// A warp sends tile j+1 as soon as it has received and read tile j; flow control is
// implicit (the peer sent tile j only after reading tile j-1 from the buffer that tile
// j+1 goes to), so two buffers per warp suffice.
//
// Tensor memory (496 of 512 columns): O half (256 fp32), S (64 fp32), P (32 columns
// of packed bf16 pairs) and this CTA's Q slice (144 columns of bf16 pairs), so both
// products read one operand from TMEM: S = Q.K^T and O += P.V are TS-form tcgen05.mma.
// Shared memory: a 4-stage ring of 64-key tiles (4 x 8 KB of ckv in 128-byte swizzle,
// 4 KB of kpe in 64-byte swizzle per stage), two partial-S exchange buffers (2 x 24 KB)
// that the peer fills, and small reduction buffers.
//
// Warp roles (384 threads per CTA; 352 in the instance for packed tokens on whole pages):
//   warps 0-7  softmax / correction / epilogue / Q loading.  Warp w serves TMEM lanes
//              32*(w%4) .. +31 (lane = query head) and key columns 32*(w/4) .. +31 of
//              each tile; the two warps of a lane group combine their row maxima through
//              shared memory and a 64-thread named barrier.  The loop is software
//              pipelined: tile j+1's partial S leaves for the peer before tile j's
//              softmax runs, and tile j+2's S is being computed meanwhile.
//   warp 8     producer: one TMA box load per column chunk when the tile's 64 slots
//              are contiguous (a whole page of 64); otherwise every lane copies
//              16-byte pieces of the gathered rows with cp.async into the same
//              swizzled layout (TMA's row gather was measured slower).  Keys past the
//              row's length are zero-filled.
//   warp 9     issues S = Q.K^T (one thread) and owns TMEM
//   warp 10    issues O += P.V (one thread); tcgen05.mma issue blocks while the tensor
//              pipe is busy, so the two products get separate issuing threads.
//   warp 11    second copy warp of the small-page and FP8 instances (each copy warp
//              takes 32 of a tile's 64 keys); idle in the whole-page instance.
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "tc_kernel.h"

namespace mla {

using namespace ptx;

namespace {

constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;    // issues S = Q.K^T; owns TMEM
constexpr int kPvWarp = 10;    // issues O += P.V
// The small-page instance has a second copy warp: a copied tile's keys are split
// between the two warps (32 each).
constexpr int kCopyWarp2 = 11;
// Threads of an instance.  The page-aligned instance without packed tokens has an idle
// twelfth warp: with it the compiled softmax loop runs measurably faster (prefill ~8%),
// while the packed-token instance is faster with eleven.
template <bool kGather, bool kPack>
constexpr int instance_threads() { return kGather || !kPack ? 384 : 352; }
constexpr int kStages = 4;
constexpr int kQkSteps = 18;                // 288-wide depth slice / 16
constexpr uint32_t kChunkKV = 64 * 128;     // 64 rows x 64 bf16, 128-byte swizzle
constexpr uint32_t kChunkPe = 64 * 64;      // 64 rows x 32 bf16, 64-byte swizzle
constexpr uint32_t kStageBytes = 4 * kChunkKV + kChunkPe;
constexpr uint32_t kXBytes = 128 * 64 * 3;  // one partial-S tile, 24-bit floats
constexpr uint32_t kOffKV = 0;
constexpr uint32_t kOffX = kOffKV + kStages * kStageBytes;
constexpr uint32_t kXWarpBytes = kXBytes / 8;  // one softmax warp's piece: 32 rows x 32 keys
constexpr uint32_t kOffRed = kOffX + 2 * kXBytes;  // [2][2][128] row maxima
constexpr uint32_t kOffL = kOffRed + 2 * 2 * 128 * 4;  // [2][128] row sums
constexpr uint32_t kOffStg = kOffL + 2 * 128 * 4;  // [softmax warp] 2 KB: Q in / O out transposes
constexpr uint32_t kOffDesc = kOffStg + 8 * 2048;  // ring of kDescRing tile descriptors
constexpr int kDescRing = 8;
constexpr uint32_t kOffBar = kOffDesc + kDescRing * 40;
constexpr uint32_t kOffMisc = kOffBar + 512;
constexpr uint32_t kSmemBytes = kOffMisc + 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // 256 columns
constexpr uint32_t kColS = 256;  // 64 columns
constexpr uint32_t kColP = 320;  // 32 columns
constexpr uint32_t kColQ = 352;  // 144 columns
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by more than 2^8

enum Bar : uint32_t {
  Q_FULL, KV_FULL0, KV_EMPTY0 = KV_FULL0 + kStages, S_FULL = KV_EMPTY0 + kStages, S_EMPTY, P_FULL, PV_DONE,
  X_FULL0, O_FULL = X_FULL0 + 16, O_EMPTY, DRAIN, DESC0,
  RAW0,  // FP8 instance: a stage's raw bytes have landed (one per stage)
  NUM_BARS = RAW0 + kStages
};

// Dequantised FP8 latent values of 8 keys (keys k0 .. k0 + 7 of the tile): lane l holds
// each key's 8 E4M3 codes raw[i] and its scale sc[i] and stores the 8 scaled bf16 values
// at row k of the chunk at dst_chunk (128-byte rows, 16-byte unit cu swizzled by k & 7),
// the layout the bf16 copies write.
__device__ __forceinline__ void fp8_store_latent(const uint2 (&raw)[8], const float (&sc)[8], uint32_t dst_chunk,
                                                 int k0, uint32_t cu) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int k = k0 + i;
    const uint4 v = ptx::e4m3x8_scaled_to_bf16x8(raw[i], sc[i]);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst_chunk + k * 128 + ((cu ^ (k & 7)) << 4)),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
}

// The two softmax warps that serve the same TMEM lanes (w and w + 4) meet at a named
// barrier.  A warp leaves the softmax loop early only after some wait gave up, which
// raises the abort flag first; on leaving it arrives once at its pair barrier, which
// releases a partner waiting there, and every warp reads the flag right after each
// pair barrier and leaves too, so no warp waits at a pair barrier for ever.
__device__ __forceinline__ void pair_sync(int warp) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
}
__device__ __forceinline__ void pair_release(int warp) {
  asm volatile("bar.arrive %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
}

struct Misc {
  uint32_t tmem;
  int abort;
  long long C;  // cost units of the call (0: no tiles)
  Cursor cur;
};

static_assert(NUM_BARS * 8 <= 512, "barrier area");
static_assert(sizeof(Misc) <= 64, "misc area");
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kStageBytes % 1024 == 0, "stage alignment");

// Partial scores cross between the two CTAs as 24-bit floats: the fp32 value rounded
// to nearest at 16 significant bits (relative error <= 2^-16), four values in three words.
// Both CTAs add the rounded values, so their scores stay bitwise identical.
// round24: add half of the dropped byte (a carry rounds up into the exponent); pack24
// then keeps the top three bytes of each value, so the pair rounds to nearest.
__device__ __forceinline__ uint32_t round24(uint32_t f) { return f + 0x80u; }

__device__ __forceinline__ void pack24(const uint32_t* v, uint32_t* w) {  // v[4] -> w[3], byte permutes
  w[0] = __byte_perm(v[0], v[1], 0x5321);  // v0.b1 v0.b2 v0.b3 v1.b1
  w[1] = __byte_perm(v[1], v[2], 0x6532);  // v1.b2 v1.b3 v2.b1 v2.b2
  w[2] = __byte_perm(v[2], v[3], 0x7653);  // v2.b3 v3.b1 v3.b2 v3.b3
}

__device__ __forceinline__ void unpack24(const uint32_t* w, float* x) {  // w[3] -> x[4], low bytes zero
  x[0] = __uint_as_float(__byte_perm(w[0], 0u, 0x2104));
  x[1] = __uint_as_float(__funnelshift_r(w[0], w[1], 16) & 0xFFFFFF00u);
  x[2] = __uint_as_float(__funnelshift_r(w[1], w[2], 8) & 0xFFFFFF00u);
  x[3] = __uint_as_float(__byte_perm(w[2], 0u, 0x3214));
}

// A warp's 2 KB transpose buffer holds 32 rows x 64 bytes: 16-byte chunk c of row r sits
// in slot 4r + (c ^ ((r >> 1) & 3)), so both a row-per-lane access (lane r, chunks 0..3)
// and a coalesced access (lanes 4k..4k+3 on the four chunks of one row) are free of bank
// conflicts.
__device__ __forceinline__ uint32_t stg_slot(int r, int c) { return 16u * (4 * r + (c ^ ((r >> 1) & 3))); }


// Tiles of a worker in order, with their segment.
struct TileIter {
  Walker walk;
  Segment seg;
  int t;
  int nseg;  // index of seg among the worker's segments
  bool live;
  __device__ void init(const PlanArgs& pa, const Cursor& c) {
    walk.init(pa, c);
    nseg = -1;
    live = walk.next(seg);
    if (live) {
      t = seg.t_begin;
      nseg = 0;
    }
  }
  __device__ bool first() const { return t == seg.t_begin; }
  __device__ bool last() const { return t == seg.t_end - 1; }
  __device__ void advance() {
    if (++t == seg.t_end) {
      live = walk.next(seg);
      if (live) {
        t = seg.t_begin;
        ++nseg;
      }
    }
  }
};

// What the MMA and softmax roles need to know about one tile; written by the
// producer into a ring of kDescRing entries (slot j % kDescRing) before it issues the
// tile's loads, and read after the tile's KV_FULL barrier has completed.  A slot is
// rewritten only for tile j + kDescRing, i.e. after P.V of tile j + kDescRing - kStages,
// by which time every reader of tile j is done with it.
struct TileDesc {
  int t;              // tile within the query row
  int len;            // keys the row sees
  int row;            // query row (decode: request)
  int next_row;       // query row of the next segment when kLast, else -1
  int slot;           // partial-result slot of the segment
  int flags;          // kFirst | kLast | kWhole | kCopied (loaded by cp.async, not TMA)
  int nseg;           // index of the segment among this worker's segments
  int pad;
  // Bit k: key k of the tile is one of the row's keys and names a slot of the cache
  // (keys past the row's length, padding entries and out-of-range slots are skipped).
  unsigned long long valid;
};
constexpr int kFirst = 1, kLast = 2, kWhole = 4, kCopied = 8;
static_assert(sizeof(TileDesc) == 40, "descriptor size");

}  // namespace

// kGather: the cache's pages are smaller than a tile (page size not a multiple of 64),
// so tiles are copied slot by slot and the producer reads slot ids a tile ahead.
// kPack: packed multi-token decode; TMEM lane m holds token m / mtp_h, head m % mtp_h of
// the request, and each token's causal horizon masks the scores lane by lane.
template <bool kGather, bool kPack, bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(instance_threads<kGather, kPack>(), 1)
    mla_tc_kernel(const __grid_constant__ TmaMaps maps, const MlaParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  Misc& misc = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int w = blockIdx.x >> 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort = &misc.abort;
  const unsigned long long wait_ns = p.wait_ns;  // limit of every bounded wait
  auto bar = [&](uint32_t i) { return sbase + kOffBar + 8u * i; };

  if (threadIdx.x == 0) {
    misc.abort = (sbase & 1023u) ? 1 : 0;  // swizzled tiles need 1 KB alignment
    if (misc.abort) atomicOr(p.status, kStatusInternal);
    mbar_init(bar(Q_FULL), kSoftmaxWarps);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(KV_FULL0 + s), kGather ? 2 : 1);  // one arrival per copy warp
      mbar_init(bar(KV_EMPTY0 + s), 1);
    }
    mbar_init(bar(S_FULL), 1);
    mbar_init(bar(S_EMPTY), kSoftmaxWarps);
    mbar_init(bar(P_FULL), kSoftmaxWarps);
    mbar_init(bar(PV_DONE), 1);
    for (int i = 0; i < 16; ++i) mbar_init(bar(X_FULL0 + i), 1);  // [buffer][softmax warp]
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(O_EMPTY), kSoftmaxWarps);
    mbar_init(bar(DRAIN), 2);  // one commit from each MMA-issuing thread
    mbar_init(bar(DESC0), 1);  // the first tile's descriptor is written
    if (kFp8)
      for (int s = 0; s < kStages; ++s) mbar_init(bar(RAW0 + s), 2);  // one arrival per copy warp
    fence_mbar_init();
    // Arm the first phase of every exchange barrier before the peer can send.
    for (int i = 0; i < 16; ++i) mbar_arrive_expect_tx(bar(X_FULL0 + i), kXWarpBytes);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + kOffMisc, kTmemCols);  // misc.tmem is the first word of Misc
    tmem_relinquish();
  }
  const PlanArgs pa{p.kv_indptr, p.qo_indptr, p.batch, p.num_kv_indices, p.topk};
  if (warp == 0) {
    Cursor c;
    const long long C = warp_plan(pa, w, p.workers, &c);
    if (lane == 0) {
      misc.cur = c;
      misc.C = C;
      // Start pulling the first query row into L2 now; the softmax warps read it into
      // TMEM as soon as the first tile's descriptor exists.  (If that row turns out to
      // have no keys, the prefetch was merely useless.)
      if (c.g < c.g_end && c.b < p.batch) {
        const int row = p.qo_indptr ? __ldg(p.qo_indptr + c.b) + c.i : c.b;
        if (row >= 0 && row < p.rows) {
          if (rank == 0) bulk_prefetch_l2(p.q_nope + (size_t)row * p.heads * kDimCkv, p.heads * kDimCkv * 2);
          else bulk_prefetch_l2(p.q_pe + (size_t)row * p.heads * kDimKpe, p.heads * kDimKpe * 2);
        }
      }
    }
    if (w == 0 && rank == 0) warp_write_empty_rows(p);
    // This worker's row of merge counters starts every call at zero: the merge kernel
    // counts on it only after this grid has completed, so no state is carried from call
    // to call (nor from a call with another worker count or head count).
    if (rank == 0)
      for (int g = lane; g < (p.heads + 7) / 8; g += 32) p.merge_count[(size_t)w * ((p.heads + 7) / 8) + g] = 0;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = misc.tmem;
  const long long C = misc.C;
  Cursor cur = misc.cur;
  if (misc.abort) cur.g_end = cur.g;  // no work

  if (warp == kProducerWarp || (kGather && warp == kCopyWarp2)) {
    const int part = kGather && warp == kCopyWarp2 ? 1 : 0;  // copy warp index
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      if constexpr (kFp8) {
        prefetch_tensormap(&maps.f8_lat);
        prefetch_tensormap(&maps.f8_scl);
        prefetch_tensormap(&maps.f8_rope);
      } else {
        prefetch_tensormap(&maps.ckv);
        prefetch_tensormap(&maps.kpe);
      }
    }
    // Slot ids of tile t of a segment: lanes hold keys lane and lane + 32; keys past
    // the row's length get a slot outside the cache (TMA reads zeros there).  A TMA tile
    // takes a few instructions, so its ids are loaded just before the wait for its stage;
    // with small pages (kGather) a copied tile's copies take long to issue, so the next
    // tile's ids (same row) are loaded before them and are ready when that tile comes up.
    auto eval_slots = [&](int nvalid, int s0, int s1, bool& contiguous, int& first, unsigned long long& valid) {
      first = __shfl_sync(0xffffffffu, s0, 0);
      const bool run = nvalid == kTileKeys && s0 == first + lane && s1 == first + lane + 32 && first >= 0 &&
                       first <= p.num_slots - kTileKeys;
      contiguous = __all_sync(0xffffffffu, run);
      // Keys past the row's length carry slot num_slots, so the range test covers them.
      const unsigned lo = __ballot_sync(0xffffffffu, s0 >= 0 && s0 < p.num_slots);
      const unsigned hi = __ballot_sync(0xffffffffu, s1 >= 0 && s1 < p.num_slots);
      valid = (unsigned long long)lo | ((unsigned long long)hi << 32);
    };
    auto tile_slots = [&](const Segment& sg, int t, int& s0, int& s1, bool& contiguous, int& first,
                          unsigned long long& valid) {
      const int key0 = t * kTileKeys;
      const int nvalid = min(kTileKeys, sg.len - key0);
      const int* ip = p.kv_indices + sg.kv0 + key0;
      s0 = lane < nvalid ? __ldg(ip + lane) : p.num_slots;
      s1 = lane + 32 < nvalid ? __ldg(ip + lane + 32) : p.num_slots;
      eval_slots(nvalid, s0, s1, contiguous, first, valid);
    };
    const bool decode = p.qo_indptr == nullptr;
    const uint64_t kv_policy = l2_policy_evict_first();
    const int ckv_col = (int)rank * 256;
    const int kpe_col = (int)rank * 32;
    TileIter it;
    it.init(pa, cur);
    TileDesc* desc = reinterpret_cast<TileDesc*>(smem + kOffDesc);
    const bool fault_worker = p.fault_skip_tile >= 1 && w == 0 && rank == 0;
    uint32_t j = 0;
    bool have_next = false;  // next_s0/next_s1 hold this tile's ids, loaded a tile ago
    int next_s0 = 0, next_s1 = 0;
    if constexpr (kFp8) {
      // ---- FP8 cache.  Copy warps 8 and 11 (part 0 / 1) each own 32 keys of every tile.
      // For tile j a warp issues the tile's raw bytes into the stage as staging -- TMA
      // boxes for a run of 64 slots (latent halves, scales, and the rope half straight to
      // its place), cp.async otherwise -- then dequantises tile j - 1 from its staging into
      // the bf16 layout the MMA reads: one tile of lag keeps a tile's loads in flight while
      // the previous one is converted.  A warp's staging lies inside the rows it writes
      // (half `part` of every 8 KB chunk): the two 128-byte halves of key k's latent sit in
      // row k of chunks 2 and 3 -- the rows key k's bf16 values replace -- and the warp's
      // 32 keys' scales in its rows 24 .. 27 of chunk 1, which only the last group of keys
      // overwrites.  Converting 8 keys at a time (group g writes rows 8g .. 8g + 7) thus
      // never overwrites staging it has not read, and the two warps never wait for each
      // other.
      const uint32_t half_off = (uint32_t)part * 4096u;
      auto stage_addr = [&](uint32_t t) { return sbase + kOffKV + (t % kStages) * kStageBytes; };
      auto convert = [&](uint32_t t) -> bool {
        if (!mbar_wait(bar(RAW0 + t % kStages), (t / kStages) & 1, abort, p.status, kStatusTimeout, wait_ns))
          return false;
        const uint32_t S = stage_addr(t);
        // Lane l's 8 codes of key kk: latent bytes 8l .. 8l + 7, in chunk 2 + l / 16.
        const uint32_t lat_s = S + (2 + (lane >> 4)) * kChunkKV + half_off + 8 * (lane & 15);
        const uint32_t scl_s = S + kChunkKV + half_off + 3072 + 4 * (2 * rank + (lane >> 4));
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint2 raw[8];
          float sc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int kk = 8 * g + i;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(raw[i].x), "=r"(raw[i].y) : "r"(lat_s + kk * 128)
                         : "memory");
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sc[i]) : "r"(scl_s + kk * 16) : "memory");
          }
          __syncwarp();
          fp8_store_latent(raw, sc, S + (uint32_t)(lane >> 3) * kChunkKV, 32 * part + 8 * g, lane & 7);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KV_FULL0 + t % kStages));  // (release: orders the stores)
        return true;
      };
      uint32_t issued = 0;  // tiles whose raw bytes were requested
      bool fok = true;
      for (; it.live; it.advance(), ++j) {
        const int stage = j % kStages;
        int s0, s1, first;
        bool contiguous;
        unsigned long long valid;
        if (have_next) {
          s0 = next_s0;
          s1 = next_s1;
          eval_slots(min(kTileKeys, it.seg.len - it.t * kTileKeys), s0, s1, contiguous, first, valid);
          have_next = false;
        } else {
          tile_slots(it.seg, it.t, s0, s1, contiguous, first, valid);
        }
        if (j >= kStages &&
            !mbar_wait(bar(KV_EMPTY0 + stage), ((j / kStages) - 1) & 1, abort, p.status, kStatusTimeout, wait_ns)) {
          fok = false;
          break;
        }
        const uint32_t S = stage_addr(j);
        const uint32_t rawbar = bar(RAW0 + stage);
        const bool skip = fault_worker && (int)j == p.fault_skip_tile;
        if (lane == 0 && part == 0) {
          TileDesc d;
          d.t = it.t;
          d.len = it.seg.len;
          d.row = it.seg.row;
          d.slot = it.seg.slot;
          d.nseg = it.nseg;
          d.flags = (it.first() ? kFirst : 0) | (it.last() ? kLast : 0) | (it.seg.whole ? kWhole : 0) | kCopied;
          d.next_row = -1;
          d.pad = 0;
          d.valid = valid;
          if (it.last()) {
            TileIter peek = it;
            peek.advance();
            if (peek.live) {
              d.next_row = peek.seg.row;
              const size_t r = (size_t)d.next_row * p.heads;
              if (rank == 0) bulk_prefetch_l2(p.q_nope + r * kDimCkv, p.heads * kDimCkv * 2);
              else bulk_prefetch_l2(p.q_pe + r * kDimKpe, p.heads * kDimKpe * 2);
            }
          }
          desc[j % kDescRing] = d;
          if (j == 0) mbar_arrive(bar(DESC0));
        }
        __syncwarp();
        if (skip) {
          // Test of the give-up path: this tile's bytes are never requested.
        } else if (contiguous) {
          if (lane == 0) {
            if (part == 0) {
              fence_proxy_async_smem();  // the stage last held bf16 written by the generic proxy
              mbar_arrive_expect_tx(rawbar, 2 * 8192 + 2 * 512 + 64 * 64);
#pragma unroll
              for (int h = 0; h < 2; ++h)  // latent bytes 128h .. 128h + 127 of the CTA's half: chunk 2 + h
                tma_load_2d(S + (2 + h) * kChunkKV, &maps.f8_lat, 256 * (int)rank + 128 * h, first, rawbar);
#pragma unroll
              for (int h = 0; h < 2; ++h)  // scales of keys 32h .. 32h + 31: chunk 1, rows 32h + 24 ..
                tma_load_2d(S + kChunkKV + h * 4096 + 3072, &maps.f8_scl, 512, first + 32 * h, rawbar);
              tma_load_2d(S + 4 * kChunkKV, &maps.f8_rope, 528 + 64 * (int)rank, first, rawbar);
            } else {
              mbar_arrive(rawbar);
            }
          }
        } else {
          if (!it.last()) {  // the next tile of this row: its slot ids a tile ahead
            const int key1 = (it.t + 1) * kTileKeys;
            const int nv1 = min(kTileKeys, it.seg.len - key1);
            const int* ip1 = p.kv_indices + it.seg.kv0 + key1;
            next_s0 = lane < nv1 ? __ldg(ip1 + lane) : p.num_slots;
            next_s1 = lane + 32 < nv1 ? __ldg(ip1 + lane + 32) : p.num_slots;
            have_next = true;
          }
          const int sp = part ? s1 : s0;
          const uint8_t* tok = p.kv_fp8;
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {  // two keys per instruction: 16 lanes x 16 bytes each
            const int kk = 2 * i + (lane >> 4);
            const int slot = __shfl_sync(0xffffffffu, sp, kk);
            const bool okk = slot >= 0 && slot < p.num_slots;
            cp_async_16_zfill(S + (2 + ((lane & 15) >> 3)) * kChunkKV + half_off + kk * 128 + 16 * (lane & 7),
                              tok + (okk ? (size_t)slot * kFp8TokenBytes + 256 * rank + 16 * (lane & 15) : 0),
                              okk ? 16 : 0);
          }
          {  // the four scales of key `lane`
            const bool okk = sp >= 0 && sp < p.num_slots;
            cp_async_16_zfill(S + kChunkKV + half_off + 3072 + lane * 16,
                              tok + (okk ? (size_t)sp * kFp8TokenBytes + 512 : 0),
                              okk ? 16 : 0);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // the rope half, into its place
            const int kk = 8 * i + (lane >> 2), k = 32 * part + kk;
            const int slot = __shfl_sync(0xffffffffu, sp, kk);
            const bool okk = slot >= 0 && slot < p.num_slots;
            cp_async_16_zfill(S + 4 * kChunkKV + k * 64 + (((lane & 3) ^ ((k >> 1) & 3)) << 4),
                              tok + (okk ? (size_t)slot * kFp8TokenBytes + 528 + 64 * rank + (lane & 3) * 16 : 0),
                              okk ? 16 : 0);
          }
          cp_async_mbar_arrive(rawbar);
          __syncwarp();
          if (lane == 0) mbar_arrive(rawbar);
        }
        __syncwarp();
        issued = j + 1;
        if (j >= 1 && !convert(j - 1)) {
          fok = false;
          break;
        }
      }
      if (fok && issued >= 1) convert(issued - 1);
      // Drain: wait (bounded) for the last raw request of every stage, so no copy is in
      // flight when the CTA exits, whatever happened above.
      if (lane == 0) {
        volatile int no_abort = 0;
        for (uint32_t s = 0; s < kStages && s < issued; ++s) {
          const uint32_t last = issued - 1 - ((issued - 1 - s) % kStages);
          if (fault_worker && (int)last == p.fault_skip_tile) continue;  // never requested
          mbar_wait(bar(RAW0 + (last % kStages)), (last / kStages) & 1, &no_abort, p.status, kStatusTimeout,
                    wait_ns);
        }
      }
    } else {
    for (; it.live; it.advance(), ++j) {
      const int stage = j % kStages;
      int s0, s1, first;
      bool contiguous;
      unsigned long long valid;
      if (kGather && have_next) {
        s0 = next_s0;
        s1 = next_s1;
        eval_slots(min(kTileKeys, it.seg.len - it.t * kTileKeys), s0, s1, contiguous, first, valid);
        have_next = false;
      } else {
        // Slot ids first, so their load overlaps the wait for a free stage.
        tile_slots(it.seg, it.t, s0, s1, contiguous, first, valid);
      }
      if (j >= kStages &&
          !mbar_wait(bar(KV_EMPTY0 + stage), ((j / kStages) - 1) & 1, abort, p.status, kStatusTimeout, wait_ns))
        break;
      const uint32_t kvbar = bar(KV_FULL0 + stage);
      const uint32_t dst = sbase + kOffKV + stage * kStageBytes;
      const bool skip = fault_worker && (int)j == p.fault_skip_tile;
      if (lane == 0 && part == 0) {
        TileDesc d;
        d.t = it.t;
        d.len = it.seg.len;
        d.row = it.seg.row;
        d.slot = it.seg.slot;
        d.nseg = it.nseg;
        d.flags = (it.first() ? kFirst : 0) | (it.last() ? kLast : 0) | (it.seg.whole ? kWhole : 0) |
                  (contiguous ? 0 : kCopied);
        d.next_row = -1;
        d.pad = 0;
        d.valid = valid;
        if (it.last()) {
          TileIter peek = it;
          peek.advance();
          if (peek.live) {
            d.next_row = peek.seg.row;
            // The softmax warps load that row's Q into TMEM once this tile's QK is done,
            // a few tiles from now; pull it into L2 meanwhile.
            const size_t r = (size_t)d.next_row * p.heads;
            if (rank == 0) bulk_prefetch_l2(p.q_nope + r * kDimCkv, p.heads * kDimCkv * 2);
            else bulk_prefetch_l2(p.q_pe + r * kDimKpe, p.heads * kDimKpe * 2);
          }
        }
        desc[j % kDescRing] = d;
        if (j == 0) mbar_arrive(bar(DESC0));  // lets the softmax warps load Q early
        // TMA tile: the one arrival, with the tile's bytes (release: orders the descriptor
        // before the tile).  Copied tile: lane 0 arrives after the lanes' copies below.
        if (contiguous && !skip) mbar_arrive_expect_tx(kvbar, kStageBytes);
      }
      __syncwarp();
      if (skip) {
        // Test of the give-up path: this tile is never loaded and never arrives, so every
        // wait on it runs into its limit.
      } else if (contiguous) {
        if (kGather && part == 1) {
          if (lane == 0) mbar_arrive(kvbar);
        } else if (lane == 0) {
          if (decode) {  // each KV byte is read once: evict it first
            for (int c = 0; c < 4; ++c)
              tma_load_2d_hint(dst + c * kChunkKV, &maps.ckv, ckv_col + c * 64, first, kvbar, kv_policy);
            tma_load_2d_hint(dst + 4 * kChunkKV, &maps.kpe, kpe_col, first, kvbar, kv_policy);
          } else {  // prefill rows of a request share its KV tiles through L2
            for (int c = 0; c < 4; ++c) tma_load_2d(dst + c * kChunkKV, &maps.ckv, ckv_col + c * 64, first, kvbar);
            tma_load_2d(dst + 4 * kChunkKV, &maps.kpe, kpe_col, first, kvbar);
          }
        }
      } else {
        // Scattered slots: each key's 512-byte ckv half-row is one warp-wide 16-byte
        // cp.async per lane; the kpe rows go eight keys per instruction.  The shared
        // addresses follow the 128-byte (ckv) and 64-byte (kpe) swizzles the MMA
        // descriptors expect.  Keys past the row's length and slots outside the cache
        // are zero-filled.
        if (kGather && !it.last()) {  // the next tile of this row
          const int key1 = (it.t + 1) * kTileKeys;
          const int nv1 = min(kTileKeys, it.seg.len - key1);
          const int* ip1 = p.kv_indices + it.seg.kv0 + key1;
          next_s0 = lane < nv1 ? __ldg(ip1 + lane) : p.num_slots;
          next_s1 = lane + 32 < nv1 ? __ldg(ip1 + lane + 32) : p.num_slots;
          have_next = true;
        }
        const char* ckv_src = reinterpret_cast<const char*>(p.ckv + ckv_col) + lane * 16;
        const uint32_t cu = lane & 7, cc = lane >> 3;
        const char* kpe_src = reinterpret_cast<const char*>(p.kpe + kpe_col) + (lane & 3) * 16;
        if constexpr (kGather) {  // this warp's 32 keys: part * 32 .. + 31
          const int sp = part ? s1 : s0;
#pragma unroll 8
          for (int kk = 0; kk < 32; ++kk) {
            const int k = 32 * part + kk;
            const int slot = __shfl_sync(0xffffffffu, sp, kk);
            const bool okk = slot >= 0 && slot < p.num_slots;
            cp_async_16_zfill(dst + cc * kChunkKV + k * 128 + ((cu ^ (k & 7)) << 4),
                              ckv_src + (okk ? (size_t)slot * (kDimCkv * 2) : 0), okk ? 16 : 0);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kk = 8 * i + (lane >> 2), k = 32 * part + kk;
            const int slot = __shfl_sync(0xffffffffu, sp, kk);
            const bool okk = slot >= 0 && slot < p.num_slots;
            cp_async_16_zfill(dst + 4 * kChunkKV + k * 64 + (((lane & 3) ^ ((k >> 1) & 3)) << 4),
                              kpe_src + (okk ? (size_t)slot * (kDimKpe * 2) : 0), okk ? 16 : 0);
          }
        } else {
#pragma unroll 8
          for (int k = 0; k < kTileKeys; ++k) {
            const int slot = __shfl_sync(0xffffffffu, k < 32 ? s0 : s1, k & 31);
            const bool okk = slot >= 0 && slot < p.num_slots;
            cp_async_16_zfill(dst + cc * kChunkKV + k * 128 + ((cu ^ (k & 7)) << 4),
                              ckv_src + (okk ? (size_t)slot * (kDimCkv * 2) : 0), okk ? 16 : 0);
          }
#pragma unroll
          for (int i = 0; i < kTileKeys / 8; ++i) {
            const int k = 8 * i + (lane >> 2);
            const int slot = __shfl_sync(0xffffffffu, i < 4 ? s0 : s1, k & 31);
            const bool okk = slot >= 0 && slot < p.num_slots;
            cp_async_16_zfill(dst + 4 * kChunkKV + k * 64 + (((lane & 3) ^ ((k >> 1) & 3)) << 4),
                              kpe_src + (okk ? (size_t)slot * (kDimKpe * 2) : 0), okk ? 16 : 0);
          }
        }
        cp_async_mbar_arrive(kvbar);
        __syncwarp();
        if (lane == 0) mbar_arrive(kvbar);
      }
      __syncwarp();
    }
    // Drain: wait (bounded) for the last load into every stage, so no copy is in
    // flight when the CTA exits, whatever happened above.
    if (lane == 0) {
      volatile int no_abort = 0;
      for (uint32_t s = 0; s < kStages && s < j; ++s) {
        const uint32_t last = j - 1 - ((j - 1 - s) % kStages);
        if (fault_worker && (int)last == p.fault_skip_tile) continue;  // never issued
        mbar_wait(bar(KV_FULL0 + (last % kStages)), (last / kStages) & 1, &no_abort, p.status, kStatusTimeout, wait_ns);
      }
    }
    }  // bf16 caches
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ------------------------------------------------------------ MMA issuers
    // tcgen05.mma issue blocks while the tensor pipe is busy, so QK and PV come from
    // two threads: PV(j) goes out as soon as P(j) exists instead of queueing behind the
    // issue of a later QK, which frees the tile's stage for the producer sooner.
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);
      const TileDesc* desc = reinterpret_cast<const TileDesc*>(smem + kOffDesc);
      const uint32_t ntiles = (uint32_t)(cur.g_end - cur.g);
      if (warp == kMmaWarp) {
        // S = Q . K^T for every tile (TS form: Q slice in TMEM, K tile in shared memory).
        for (uint32_t jq = 0; jq < ntiles; ++jq) {
          const uint32_t stage = jq % kStages;
          if (!mbar_wait(bar(KV_FULL0 + stage), (jq / kStages) & 1, abort, p.status, kStatusTimeout, wait_ns)) break;
          const TileDesc d = desc[jq % kDescRing];
          if (((d.flags & kFirst) && !mbar_wait(bar(Q_FULL), d.nseg & 1, abort, p.status, kStatusTimeout, wait_ns)) ||
              (jq >= 1 && !mbar_wait(bar(S_EMPTY), (jq - 1) & 1, abort, p.status, kStatusTimeout, wait_ns)))
            break;
          if (d.flags & kCopied) fence_proxy_async_smem();  // written through the generic proxy
          tc_fence_after();
          const uint32_t kv = sbase + kOffKV + stage * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kQkSteps; ++kk) {
            const uint64_t b = kk < 16 ? smem_desc_sw128(kv + (kk >> 2) * kChunkKV + (kk & 3) * 32, 16, 1024)
                                       : smem_desc_sw64(kv + 4 * kChunkKV + (kk - 16) * 32, 16, 512);
            mma_bf16_ts(tmem + kColS, tmem + kColQ + 8 * kk, b, kIdescQK, kk != 0 ? 1u : 0u);
          }
          mma_commit(bar(S_FULL));
        }
      } else {
        // This thread idles until the first P exists: write the worker's merge record.
        if (rank == 0) {
          TileIter first;
          first.init(pa, cur);
          p.records[w] = make_record(first.live, first.seg, C, p.workers);
        }
        // O += P . V for every tile (TS form: P in TMEM, V = the ckv half of the tile).
        // The tile's descriptor is visible here: the softmax warps read it after the
        // tile's KV_FULL and only then arrive on P_FULL.
        for (uint32_t jv = 0; jv < ntiles; ++jv) {
          const uint32_t stage = jv % kStages;
          if (!mbar_wait(bar(P_FULL), jv & 1, abort, p.status, kStatusTimeout, wait_ns)) break;
          const TileDesc d = desc[jv % kDescRing];
          const bool first = d.flags & kFirst;
          if (first && d.nseg > 0 && !mbar_wait(bar(O_EMPTY), (d.nseg - 1) & 1, abort, p.status, kStatusTimeout, wait_ns))
            break;
          if (d.flags & kCopied) fence_proxy_async_smem();  // written through the generic proxy
          tc_fence_after();
          const uint32_t vbase = sbase + kOffKV + stage * kStageBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t b = smem_desc_sw128(vbase + k * 2048, kChunkKV, 1024);
            mma_bf16_ts(tmem + kColO, tmem + kColP + 8 * k, b, kIdescPV, (first && k == 0) ? 0u : 1u);
          }
          mma_commit(bar(KV_EMPTY0 + stage));
          mma_commit(bar(PV_DONE));
          if (d.flags & kLast) mma_commit(bar(O_FULL));
        }
      }
      // Drain: every MMA this thread issued has completed once DRAIN fires (it counts
      // one commit from each of the two issuing threads).
      mma_commit(bar(DRAIN));
      volatile int no_abort = 0;
      mbar_wait(bar(DRAIN), 0, &no_abort, p.status, kStatusTimeout, wait_ns);
    }
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax warps
    const int row = threadIdx.x & 127;  // TMEM lane == query head
    const int half = warp >> 2;         // key columns 32*half .. +31 of each tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t x_local = sbase + kOffX;
    const uint32_t x_remote = mapa(x_local, peer);
    // Exchange piece of this warp: [buffer][warp][chunk c][lane] 16-byte units, the
    // same layout on both CTAs, so warp w of one CTA sends only to warp w of the other.
    const uint32_t piece = warp * kXWarpBytes + lane * 16;
    const uint32_t xfull_remote = mapa(bar(X_FULL0 + warp), peer);    // + 64 * buffer
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    float* lbuf = reinterpret_cast<float*>(smem + kOffL);
    const float scale = p.scale_log2;

    // This warp's transpose buffer, and the rows (query heads) it serves.
    const uint32_t stg = sbase + kOffStg + warp * 2048;
    const int row0 = (warp & 3) * 32;

    // Write the Q slice of query row `qrow` (this warp's heads, this half's depth) into
    // TMEM: half 0 -> depth 0..127 (16 x 16 B of q_nope per head), half 1 -> depth
    // 128..287 (16 x 16 B of q_nope, 4 x 16 B of q_pe).  Heads >= H get zeros.  The
    // global reads are coalesced (each instruction reads 64 contiguous bytes of eight
    // heads) and go through the transpose buffer to reach the thread that owns the head's
    // TMEM lane; all of them are issued before the first is used.
    auto write_q = [&](int qrow) {
      const int npass = half ? 5 : 4;  // 64-byte chunk groups per head
      const int hh_lo = lane >> 2, cl = lane & 3;
      uint4 v[5][4];
#pragma unroll
      for (int ps = 0; ps < 5; ++ps) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int hh = 8 * i + hh_lo;
          const int h = row0 + hh;
          v[ps][i] = make_uint4(0, 0, 0, 0);
          if (ps < npass && h < p.heads) {
            const size_t rg = (size_t)qrow * p.heads + h;
            const uint4* src =
                ps < 4 ? reinterpret_cast<const uint4*>(p.q_nope + rg * kDimCkv + rank * 256 + half * 128) + 4 * ps
                       : reinterpret_cast<const uint4*>(p.q_pe + rg * kDimKpe + rank * 32);
            v[ps][i] = __ldg(src + cl);
          }
        }
      }
      const uint32_t col = tmem + lane_base + kColQ + half * 64;
#pragma unroll
      for (int ps = 0; ps < 5; ++ps) {
        if (ps >= npass) break;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + stg_slot(8 * i + hh_lo, cl)),
                       "r"(v[ps][i].x), "r"(v[ps][i].y), "r"(v[ps][i].z), "r"(v[ps][i].w)
                       : "memory");
        __syncwarp();
        uint32_t rr[16];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(rr[4 * c]), "=r"(rr[4 * c + 1]), "=r"(rr[4 * c + 2]), "=r"(rr[4 * c + 3])
                       : "r"(stg + stg_slot(lane, c))
                       : "memory");
        __syncwarp();
        tmem_st16(col + 16 * ps, rr);  // 64 bytes = 16 columns of bf16 pairs
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Q_FULL));
    };

    // Store one 16-column slice (64 bytes per head: 4 chunks per lane in c[]) of this
    // warp's heads through the transpose buffer, so that each store instruction writes
    // 64 contiguous bytes of eight heads.  dst(h) is the slice's address for head h.
    const uint64_t keep_policy = l2_policy_evict_last();  // partials are read back by the merge
    auto store_rows = [&](const uint4 (&c)[4], auto dst, bool keep) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + stg_slot(lane, k)), "r"(c[k].x),
                     "r"(c[k].y), "r"(c[k].z), "r"(c[k].w)
                     : "memory");
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int hh = 8 * i + (lane >> 2);
        uint4 x;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                     : "r"(stg + stg_slot(hh, lane & 3))
                     : "memory");
        if (row0 + hh < p.heads) {
          if (keep) st_global_v4_hint(dst(row0 + hh) + (lane & 3), x, keep_policy);
          else dst(row0 + hh)[lane & 3] = x;
        }
      }
      __syncwarp();
    };

    const TileDesc* desc = reinterpret_cast<const TileDesc*>(smem + kOffDesc);
    const uint32_t ntiles = (uint32_t)(cur.g_end - cur.g);
    bool ok = true;
    uint32_t jf = 0;       // tiles fetched
    uint32_t nxt[24];      // own partial scores of tile jf - 1, rounded and packed
    // Fetch tile jf: read its partial S from TMEM, release S, round and pack it, and note
    // the next segment's row if this was the segment's last QK (its Q slice is written
    // after this tile's piece has left for the peer, off the exchange's critical path).
    int q_pending = -1;
    auto fetch = [&]() -> bool {
      if (!mbar_wait(bar(S_FULL), jf & 1, abort, p.status, kStatusTimeout, wait_ns)) return false;
      tc_fence_after();
      uint32_t sn[32];
      tmem_ld32(tmem + lane_base + kColS + 32 * half, sn);
      // The tile's descriptor: its KV_FULL phase has completed (QK read the tile); the
      // barrier probe overlaps the TMEM load.
      const bool kv_ok =
          mbar_wait(bar(KV_FULL0 + jf % kStages), (jf / kStages) & 1, abort, p.status, kStatusTimeout, wait_ns);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_EMPTY));  // the next QK may overwrite S now
      if (!kv_ok) return false;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        uint32_t v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = round24(sn[4 * g + e]);
        pack24(v, &nxt[3 * g]);
      }
      q_pending = desc[jf % kDescRing].next_row;
      ++jf;
      return true;
    };

    // Send this warp's piece of tile t (the packed own partial v) into the peer warp's
    // exchange buffer t & 1; the stores complete their bytes on the peer warp's X_FULL
    // barrier of that buffer.  Flow control is implicit: the piece of tile t + 1 leaves
    // only after this warp has received the peer's piece of tile t, which the peer sent
    // after it had read (and re-armed) its buffer (t + 1) & 1 for tile t - 1.
    auto send_piece = [&](uint32_t t, const uint32_t (&v)[24]) {
      const uint32_t dst = x_remote + (t & 1) * kXBytes + piece;
#pragma unroll
      for (int c = 0; c < 6; ++c)
        st_async_v4(dst + c * 512, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3], xfull_remote + 64 * (t & 1));
    };
    if (ntiles > 0) {
      if (!mbar_wait(bar(DESC0), 0, abort, p.status, kStatusTimeout, wait_ns)) {
        ok = false;
      } else {
        write_q(desc[0].row);
        ok = fetch();
        if (ok) send_piece(0, nxt);
        if (ok && q_pending >= 0) {
          write_q(q_pending);
          q_pending = -1;
        }
      }
    }
    float m_ref = -INFINITY, l = 0.f;  // l: this thread's 32 columns only
    // Packed tokens: this lane's token sees lag fewer keys than the request's last one.
    const int lag = kPack ? p.mtp_q - 1 - row / p.mtp_h : 0;
    uint32_t j = 0;
    while (ok && j < jf) {
      const TileDesc cd = desc[j % kDescRing];  // tile j (KV_FULL seen in fetch)
      const uint32_t b = j & 1;
      uint32_t own[24];  // own partial of tile j
#pragma unroll
      for (int i = 0; i < 24; ++i) own[i] = nxt[i];
      // Tile j+1's partial is fetched before this warp waits for tile j's piece, so it
      // can leave the moment tile j's has arrived.
      if (jf < ntiles && !fetch()) break;
      if (!mbar_wait<true>(bar(X_FULL0 + 8 * b + warp), (j >> 1) & 1, abort, p.status, kStatusTimeout, wait_ns)) break;
      // The peer's piece of tile j is here: load it, then send tile j+1 at once (the send
      // is what the peer waits for, so the unpacking below stays off that path).  The
      // loads are issued before the stores; the buffer is rewritten only with the peer's
      // tile j+2, which leaves the peer after tile j+1 has arrived there.
      uint32_t pw[24];
#pragma unroll
      for (int c = 0; c < 6; ++c)
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(pw[4 * c]), "=r"(pw[4 * c + 1]), "=r"(pw[4 * c + 2]), "=r"(pw[4 * c + 3])
                     : "r"(x_local + b * kXBytes + piece + c * 512)
                     : "memory");
      if (jf > j + 1) send_piece(j + 1, nxt);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(bar(X_FULL0 + 8 * b + warp), kXWarpBytes);  // arm its next use
      float s[32];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        float a[4], c4[4];
        unpack24(&own[3 * g], a);
        unpack24(&pw[3 * g], c4);
#pragma unroll
        for (int e = 0; e < 4; ++e) s[4 * g + e] = a[e] + c4[e];
      }
      if (q_pending >= 0) {
        write_q(q_pending);
        q_pending = -1;
      }
      const int nvalid = min(kTileKeys, (kPack ? cd.len - lag : cd.len) - cd.t * kTileKeys) - 32 * half;
      const uint32_t vm = static_cast<uint32_t>(cd.valid >> (32 * half));  // keys that are keys of the row
      // All 32 keys valid and a non-negative scale (the usual case): the maximum of the
      // scaled scores is the scaled maximum, and the scale folds into the exponent below.
      const bool full = nvalid >= 32 && vm == 0xffffffffu && scale >= 0.f;
      if (!full) {
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = (k < nvalid && ((vm >> k) & 1u)) ? s[k] * scale : -INFINITY;
      }
      float mx;
      {  // maximum as a tree (short dependency chains)
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(fmaxf(s[k], s[k + 8]), fmaxf(s[k + 16], s[k + 24]));
#pragma unroll
        for (int k = 0; k < 4; ++k) m8[k] = fmaxf(m8[k], m8[k + 4]);
        mx = fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3]));
      }
      if (full) mx *= scale;
      red[(b * 2 + half) * 128 + row] = mx;
      pair_sync(warp);
      if (*abort) break;
      mx = fmaxf(mx, red[(b * 2 + (half ^ 1)) * 128 + row]);
      float alpha = 1.f;
      bool rescale = false;
      if (cd.flags & kFirst) {
        m_ref = mx;
        l = 0.f;
      } else if (mx > m_ref + kRescaleLog2) {
        alpha = fast_exp2(m_ref - mx);
        m_ref = mx;
        l *= alpha;
        rescale = true;
      }
      uint32_t pk[16];
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
      // No key seen yet in this segment (m_ref = -inf: a packed token whose horizon ends
      // before the segment, or a tile of padding entries): every P is zero.
      const float mref = m_ref == -INFINITY ? 0.f : m_ref;
      if (full) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float a = fast_exp2(fmaf(s[2 * k], scale, -mref));
          const float bb = fast_exp2(fmaf(s[2 * k + 1], scale, -mref));
          sum4[k & 3] += a + bb;
          __nv_bfloat162 h = __floats2bfloat162_rn(a, bb);
          pk[k] = *reinterpret_cast<uint32_t*>(&h);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float a = fast_exp2(s[2 * k] - mref);
          const float bb = fast_exp2(s[2 * k + 1] - mref);
          sum4[k & 3] += a + bb;
          __nv_bfloat162 h = __floats2bfloat162_rn(a, bb);
          pk[k] = *reinterpret_cast<uint32_t*>(&h);
        }
      }
      l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
      // P is single-buffered: the previous tile's P.V must be done (it also settles O).
      if (j >= 1 && !mbar_wait(bar(PV_DONE), (j - 1) & 1, abort, p.status, kStatusTimeout, wait_ns)) break;
      tc_fence_after();
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          const uint32_t col = tmem + lane_base + kColO + 128 * half + 32 * cc;
          tmem_ld32(col, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(col, o);
        }
      }
      tmem_st16(tmem + lane_base + kColP + 16 * half, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_FULL));

      if (cd.flags & kLast) {
        // Epilogue: O / l to out (whole rows) or to the workspace (split rows).
        lbuf[half * 128 + row] = l;
        pair_sync(warp);
        if (*abort) break;
        const float lt = l + lbuf[(half ^ 1) * 128 + row];
        if (!mbar_wait(bar(O_FULL), cd.nseg & 1, abort, p.status, kStatusTimeout, wait_ns)) break;
        tc_fence_after();
        const float inv_l = lt > 0.f ? 1.f / lt : 0.f;  // (no key: out 0, lse -inf)
        const float lse2 = m_ref + fast_log2(lt);
        const bool valid = row < p.heads;
        const size_t frag = ((size_t)w * 2 + cd.slot) * p.heads + row;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + kColO + 128 * half + 32 * cc, o);
          tmem_ld_wait();
          const int d0 = (int)rank * 256 + 128 * half + cc * 32;
          if (cd.flags & kWhole) {
            uint4 c4[4];  // 32 columns as bf16: 64 bytes
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t wds[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(o[8 * q + 2 * e]) * inv_l,
                                                         __uint_as_float(o[8 * q + 2 * e + 1]) * inv_l);
                wds[e] = *reinterpret_cast<uint32_t*>(&h);
              }
              c4[q] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
            store_rows(c4, [&](int h) {
              return reinterpret_cast<uint4*>(p.out + ((size_t)cd.row * p.heads + h) * kDimCkv + d0);
            }, false);
          } else {
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {  // 16 fp32 columns = 64 bytes at a time
              uint4 c4[4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                c4[q] = make_uint4(__float_as_uint(__uint_as_float(o[16 * hq + 4 * q]) * inv_l),
                                   __float_as_uint(__uint_as_float(o[16 * hq + 4 * q + 1]) * inv_l),
                                   __float_as_uint(__uint_as_float(o[16 * hq + 4 * q + 2]) * inv_l),
                                   __float_as_uint(__uint_as_float(o[16 * hq + 4 * q + 3]) * inv_l));
              store_rows(c4, [&](int h) {
                return reinterpret_cast<uint4*>(p.part_o + (((size_t)w * 2 + cd.slot) * p.heads + h) * kDimCkv +
                                                d0 + 16 * hq);
              }, true);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(O_EMPTY));
        if (valid && rank == 0 && half == 0) {
          if (cd.flags & kWhole)
            p.lse[(size_t)cd.row * p.heads + row] = lse2 * 0.69314718055994531f;
          else
            p.part_lse[frag] = lse2;
        }
      }
      ++j;
    }
    // Every tile processed, or the loop left early (only ever after the abort flag was
    // raised): then release the partner, which may be waiting at the pair barrier.
    if (!ok || j < ntiles) pair_release(warp);
  }

  // The merge kernel, launched with programmatic stream serialisation, may be
  // scheduled once every CTA got here; it still waits for this grid's completion
  // (griddepcontrol.wait) before reading anything this kernel wrote.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

uint32_t tc_smem_bytes() { return kSmemBytes; }

namespace {
template <bool kGather, bool kPack, bool kFp8>
cudaError_t launch_instance(const TmaMaps& maps, const MlaParams& p, cudaStream_t stream) {
  // The shared-memory attribute is set once per device and instance; calls may come from
  // any host thread.
  static std::mutex mu;
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!configured[dev]) {
      cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel<kGather, kPack, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  mla_tc_kernel<kGather, kPack, kFp8><<<2 * p.workers, instance_threads<kGather, kPack>(), kSmemBytes, stream>>>(maps, p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_tc(const TmaMaps& maps, const MlaParams& p, bool gather, cudaStream_t stream) {
  const bool pack = p.mtp_q > 0;
  // An FP8 cache: every tile is copied and dequantised by the copy warps.
  if (p.kv_fp8) return pack ? cudaErrorInvalidValue : launch_instance<true, false, true>(maps, p, stream);
  if (gather)
    return pack ? launch_instance<true, true, false>(maps, p, stream) : launch_instance<true, false, false>(maps, p, stream);
  return pack ? launch_instance<false, true, false>(maps, p, stream) : launch_instance<false, false, false>(maps, p, stream);
}

}  // namespace mla
