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
// O[:, 256r : 256r+256] (256 columns) and loads only the key columns it needs:
//   rank 0: ckv[:, 0:256]                 (scores over dims 0..255, V for dims 0..255)
//   rank 1: ckv[:, 256:512] and kpe[:, :]  (scores over dims 256..575, V for dims 256..511)
// Each CTA computes a partial S over its depth slice; the two partial S tiles are
// swapped through distributed shared memory (st.async) and added, so every score is
// computed once and both CTAs see identical S (fp32 addition commutes), hence take
// identical softmax decisions.  This is the left/right split of the output that
// FlashMLA's "seesaw" schedule uses across two warpgroups (oL, oR), done here across
// the two SMs of a cluster with the query-key depth split as well.
//
// Warp roles (192 threads per CTA):
//   warps 0-3  softmax / correction / epilogue: thread = TMEM lane = query head
//   warp 4     TMA producer: Q tiles, and 64-key ckv/kpe tiles -- one box load per
//              column chunk when the tile's 64 slots are contiguous (a whole page of
//              64), else tile::gather4 row loads; rows past the row's length read a
//              slot index outside the cache, which TMA fills with zeros
//   warp 5     MMA issuer (one thread) and TMEM owner
// Shared memory: Q (<= 5 x 16 KB), 2 KV stages (<= 5 x 8 KB each), P (16 KB bf16),
// the partial-S exchange buffer (32 KB), mbarriers.
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "tc_kernel.h"

namespace mla {

using namespace ptx;

namespace {

constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStages = 2;
constexpr uint32_t kChunkQ = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t kChunkKV = 64 * 128;  // 64 rows x 64 bf16
constexpr uint32_t kStageBytes = 5 * kChunkKV;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + 5 * kChunkQ;
constexpr uint32_t kOffP = kOffKV + kStages * kStageBytes;
constexpr uint32_t kOffX = kOffP + 128 * 128;
constexpr uint32_t kOffBar = kOffX + 128 * 64 * 4;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;  // two 64-column S buffers
constexpr uint32_t kXBytes = 128 * 64 * 4;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8

enum Bar : uint32_t {
  Q_FULL, Q_EMPTY, KV_FULL0, KV_FULL1, KV_EMPTY0, KV_EMPTY1, S_FULL0, S_FULL1, S_EMPTY0, S_EMPTY1,
  P_FULL, PV_DONE, X_FULL, X_FREE, O_FULL, O_EMPTY, DRAIN, NUM_BARS
};

static_assert(kOffBar + NUM_BARS * 8 <= kOffBar + 256, "barrier area");
static_assert(kSmemBytes <= 232448, "shared memory");

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ TmaMaps maps, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t sh_tmem;
  __shared__ int sh_abort;
  __shared__ Cursor sh_cur;
  __shared__ long long sh_T;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int w = blockIdx.x >> 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nchunks = rank ? 5 : 4;  // Q and KV column chunks of this CTA
  volatile int* abort = &sh_abort;
  auto bar = [&](uint32_t i) { return sbase + kOffBar + 8u * i; };

  if (threadIdx.x == 0) {
    sh_abort = 0;
    mbar_init(bar(Q_FULL), 1);
    mbar_init(bar(Q_EMPTY), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(KV_FULL0 + s), 1);
      mbar_init(bar(KV_EMPTY0 + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(S_FULL0 + b), 1);
      mbar_init(bar(S_EMPTY0 + b), 4);
    }
    mbar_init(bar(P_FULL), 4);
    mbar_init(bar(PV_DONE), 1);
    mbar_init(bar(X_FULL), 1);
    mbar_init(bar(X_FREE), 4);
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(O_EMPTY), 4);
    mbar_init(bar(DRAIN), 1);
    fence_mbar_init();
    // Arm the first phase of the exchange barrier before the peer can send.
    mbar_arrive_expect_tx(bar(X_FULL), kXBytes);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sh_tmem), kTmemCols);
    tmem_relinquish();
  }
  const PlanArgs pa{p.kv_indptr, p.qo_indptr, p.batch, p.num_kv_indices};
  if (warp == 0) {
    Cursor c;
    const long long T = warp_plan(pa, w, p.workers, &c);
    if (lane == 0) {
      sh_cur = c;
      sh_T = T;
    }
    if (w == 0 && rank == 0) warp_write_empty_rows(p);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = sh_tmem;
  const long long T = sh_T;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&maps.q_nope);
      prefetch_tensormap(&maps.q_pe);
      prefetch_tensormap(&maps.ckv);
      prefetch_tensormap(&maps.kpe);
      prefetch_tensormap(&maps.ckv_g);
      prefetch_tensormap(&maps.kpe_g);
    }
    Walker walk;
    walk.init(pa, sh_cur, T, w, p.workers);
    Segment seg;
    uint32_t j = 0;
    int nseg = 0;
    int q_issued = 0;
    bool ok = true;
    while (ok && walk.next(seg)) {
      if (nseg > 0 && !mbar_wait(bar(Q_EMPTY), (nseg - 1) & 1, abort, p.status, kStatusTimeout)) break;
      ++q_issued;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(Q_FULL), nchunks * kChunkQ);
        const int qrow = seg.row * p.heads;
        for (int c = 0; c < 4; ++c)
          tma_load_2d(sbase + kOffQ + c * kChunkQ, &maps.q_nope, (int)rank * 256 + c * 64, qrow, bar(Q_FULL));
        if (rank) tma_load_2d(sbase + kOffQ + 4 * kChunkQ, &maps.q_pe, 0, qrow, bar(Q_FULL));
      }
      __syncwarp();
      for (int t = seg.t_begin; t < seg.t_end; ++t, ++j) {
        const int stage = j % kStages;
        const int key0 = t * kTileKeys;
        const int nvalid = min(kTileKeys, seg.len - key0);
        // Slot ids of the tile (read before waiting so the load overlaps the wait).
        const int* ip = p.kv_indices + seg.kv0 + key0;
        const int s0 = lane < nvalid ? __ldg(ip + lane) : p.num_slots;
        const int s1 = lane + 32 < nvalid ? __ldg(ip + lane + 32) : p.num_slots;
        if (j >= kStages &&
            !mbar_wait(bar(KV_EMPTY0 + stage), ((j / kStages) - 1) & 1, abort, p.status, kStatusTimeout)) {
          ok = false;
          break;
        }
        const int first = __shfl_sync(0xffffffffu, s0, 0);
        const bool run = nvalid == kTileKeys && s0 == first + lane && s1 == first + lane + 32 && first >= 0 &&
                         first <= p.num_slots - kTileKeys;
        const bool contiguous = __all_sync(0xffffffffu, run);
        const uint32_t kvbar = bar(KV_FULL0 + stage);
        const uint32_t dst = sbase + kOffKV + stage * kStageBytes;
        if (lane == 0) mbar_arrive_expect_tx(kvbar, nchunks * kChunkKV);
        __syncwarp();
        if (contiguous) {
          if (lane == 0) {
            for (int c = 0; c < 4; ++c)
              tma_load_2d(dst + c * kChunkKV, &maps.ckv, (int)rank * 256 + c * 64, first, kvbar);
            if (rank) tma_load_2d(dst + 4 * kChunkKV, &maps.kpe, 0, first, kvbar);
          }
        } else {
          // Lane g < 16 gathers rows 4g .. 4g+3 of the tile.
          int r[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int key = 4 * (lane & 15) + q;
            const int v0 = __shfl_sync(0xffffffffu, s0, key & 31);
            const int v1 = __shfl_sync(0xffffffffu, s1, key & 31);
            r[q] = key < 32 ? v0 : v1;
          }
          if (lane < 16) {
            for (int c = 0; c < 4; ++c)
              tma_gather4(dst + c * kChunkKV + lane * 512, &maps.ckv_g, (int)rank * 256 + c * 64, r[0], r[1], r[2],
                          r[3], kvbar);
            if (rank) tma_gather4(dst + 4 * kChunkKV + lane * 512, &maps.kpe_g, 0, r[0], r[1], r[2], r[3], kvbar);
          }
        }
        __syncwarp();
      }
      ++nseg;
    }
    // Drain: wait (bounded) for the last loads into every stage and for Q, so no copy
    // is in flight when the CTA exits, whatever happened above.
    if (lane == 0) {
      volatile int no_abort = 0;
      for (uint32_t s = 0; s < kStages && s < j; ++s) {
        const uint32_t last = j - 1 - ((j - 1 - s) % kStages);  // last tile issued into stage (last % kStages)
        mbar_wait(bar(KV_FULL0 + (last % kStages)), (last / kStages) & 1, &no_abort, p.status, kStatusTimeout);
      }
      if (q_issued > 0) mbar_wait(bar(Q_FULL), (q_issued - 1) & 1, &no_abort, p.status, kStatusTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);
      Walker walk;
      walk.init(pa, sh_cur, T, w, p.workers);
      Segment seg;
      uint32_t j = 0;
      int nseg = 0;
      bool ok = true;
      // O += P . V for global tile jj (the P of that tile is in smem).
      auto pv = [&](uint32_t jj, bool first_of_seg, int segno) -> bool {
        if (!mbar_wait(bar(P_FULL), jj & 1, abort, p.status, kStatusTimeout)) return false;
        if (first_of_seg && segno > 0 &&
            !mbar_wait(bar(O_EMPTY), (segno - 1) & 1, abort, p.status, kStatusTimeout))
          return false;
        tc_fence_after();
        const uint32_t stage = jj % kStages;
        const uint32_t vbase = sbase + kOffKV + stage * kStageBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t a = smem_desc_sw128(sbase + kOffP + k * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(vbase + k * 2048, kChunkKV, 1024);
          mma_bf16_ss(tmem + kColO, a, b, kIdescPV, (first_of_seg && k == 0) ? 0u : 1u);
        }
        mma_commit(bar(KV_EMPTY0 + stage));
        mma_commit(bar(PV_DONE));
        return true;
      };
      while (ok && walk.next(seg)) {
        if (!mbar_wait(bar(Q_FULL), nseg & 1, abort, p.status, kStatusTimeout)) break;
        for (int t = seg.t_begin; t < seg.t_end; ++t, ++j) {
          const uint32_t stage = j % kStages;
          const uint32_t buf = j & 1;
          if (!mbar_wait(bar(KV_FULL0 + stage), (j / kStages) & 1, abort, p.status, kStatusTimeout) ||
              (j >= 2 && !mbar_wait(bar(S_EMPTY0 + buf), ((j >> 1) - 1) & 1, abort, p.status, kStatusTimeout))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kvbase = sbase + kOffKV + stage * kStageBytes;
          for (int c = 0; c < nchunks; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t a = smem_desc_sw128(sbase + kOffQ + c * kChunkQ + k * 32, 16, 1024);
              const uint64_t b = smem_desc_sw128(kvbase + c * kChunkKV + k * 32, 16, 1024);
              mma_bf16_ss(tmem + kColS + 64 * buf, a, b, kIdescQK, (c | k) != 0 ? 1u : 0u);
            }
          }
          mma_commit(bar(S_FULL0 + buf));
          if (t == seg.t_end - 1) mma_commit(bar(Q_EMPTY));
          if (t > seg.t_begin && !pv(j - 1, t - 1 == seg.t_begin, nseg)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (!pv(j - 1, seg.t_end - 1 == seg.t_begin, nseg)) break;
        mma_commit(bar(O_FULL));
        ++nseg;
      }
      // Drain: every MMA issued above has completed once DRAIN fires.
      mma_commit(bar(DRAIN));
      volatile int no_abort = 0;
      mbar_wait(bar(DRAIN), 0, &no_abort, p.status, kStatusTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    const int row = threadIdx.x;  // TMEM lane == query head
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t x_local = sbase + kOffX;
    const uint32_t x_remote = mapa(x_local, peer);
    const uint32_t xfull_remote = mapa(bar(X_FULL), peer);
    const uint32_t xfree_remote = mapa(bar(X_FREE), peer);
    const uint32_t p_row = sbase + kOffP + (row >> 3) * 1024 + (row & 7) * 128;
    const float scale = p.scale_log2;
    Walker walk;
    walk.init(pa, sh_cur, T, w, p.workers);
    Segment seg, first_seg{};
    bool have_first = false;
    uint32_t j = 0;
    int nseg = 0;
    bool ok = true;
    while (ok && walk.next(seg)) {
      if (seg.first) {
        have_first = true;
        first_seg = seg;
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int t = seg.t_begin; t < seg.t_end; ++t, ++j) {
        const int nvalid = min(kTileKeys, seg.len - t * kTileKeys);
        const uint32_t buf = j & 1;
        if (!mbar_wait(bar(S_FULL0 + buf), (j >> 1) & 1, abort, p.status, kStatusTimeout)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sa[32], sb[32];
        tmem_ld32(tmem + lane_base + kColS + 64 * buf, sa);
        tmem_ld32(tmem + lane_base + kColS + 64 * buf + 32, sb);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(S_EMPTY0 + buf));
        // Swap partial scores with the peer CTA.
        if (j > 0 && !mbar_wait<true>(bar(X_FREE), (j - 1) & 1, abort, p.status, kStatusTimeout)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(x_remote + (c * 128 + row) * 16, sa[4 * c], sa[4 * c + 1], sa[4 * c + 2], sa[4 * c + 3],
                      xfull_remote);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(x_remote + ((c + 8) * 128 + row) * 16, sb[4 * c], sb[4 * c + 1], sb[4 * c + 2],
                      sb[4 * c + 3], xfull_remote);
        if (!mbar_wait<true>(bar(X_FULL), j & 1, abort, p.status, kStatusTimeout)) {
          ok = false;
          break;
        }
        float s[64];
        const float4* xin = reinterpret_cast<const float4*>(smem + kOffX);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 v = xin[c * 128 + row];
          const uint32_t* mine = c < 8 ? &sa[4 * c] : &sb[4 * (c - 8)];
          s[4 * c + 0] = __uint_as_float(mine[0]) + v.x;
          s[4 * c + 1] = __uint_as_float(mine[1]) + v.y;
          s[4 * c + 2] = __uint_as_float(mine[2]) + v.z;
          s[4 * c + 3] = __uint_as_float(mine[3]) + v.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(xfree_remote);
        if (threadIdx.x == 0) mbar_arrive_expect_tx(bar(X_FULL), kXBytes);  // arm the next phase
        // Online softmax in base 2.
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          s[k] = k < nvalid ? s[k] * scale : -INFINITY;
          mx = fmaxf(mx, s[k]);
        }
        float alpha = 1.f;
        bool rescale = false;
        if (t == seg.t_begin) {
          m_ref = mx;
        } else if (mx > m_ref + kRescaleLog2) {
          alpha = fast_exp2(m_ref - mx);
          m_ref = mx;
          l *= alpha;
          rescale = true;
        }
        uint32_t pk[32];
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float a = fast_exp2(s[2 * k] - m_ref);
          const float b = fast_exp2(s[2 * k + 1] - m_ref);
          sum += a + b;
          __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
          pk[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        l += sum;
        // The previous tile's P . V must be done before P is overwritten and O rescaled.
        if (j > 0 && !mbar_wait(bar(PV_DONE), (j - 1) & 1, abort, p.status, kStatusTimeout)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + kColO + cc * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(tmem + lane_base + kColO + cc * 32, o);
          }
          tmem_st_wait();
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = p_row + ((c ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c]), "r"(pk[4 * c + 1]),
                       "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                       : "memory");
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P_FULL));
      }
      if (!ok) break;
      // Epilogue: O / l to out (whole rows) or to the workspace (split rows).
      if (!mbar_wait(bar(O_FULL), nseg & 1, abort, p.status, kStatusTimeout)) break;
      tc_fence_after();
      const float inv_l = 1.f / l;
      const float lse2 = m_ref + fast_log2(l);
      const bool valid = row < p.heads;
      const size_t frag = ((size_t)w * 2 + seg.slot) * p.heads + row;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + kColO + cc * 32, o);
        tmem_ld_wait();
        const int d0 = (int)rank * 256 + cc * 32;
        if (valid) {
          if (seg.whole) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)seg.row * p.heads + row) * kDimCkv + d0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t wds[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(o[8 * q + 2 * e]) * inv_l,
                                                         __uint_as_float(o[8 * q + 2 * e + 1]) * inv_l);
                wds[e] = *reinterpret_cast<uint32_t*>(&h);
              }
              dst[q] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + frag * kDimCkv + d0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                   __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(O_EMPTY));
      if (valid && rank == 0) {
        if (seg.whole)
          p.lse[(size_t)seg.row * p.heads + row] = lse2 * 0.69314718055994531f;
        else
          p.part_lse[frag] = lse2;
      }
      ++nseg;
    }
    if (rank == 0 && threadIdx.x == 0) p.records[w] = make_record(have_first, first_seg, T, p.workers);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

uint32_t tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_tc(const TmaMaps& maps, const MlaParams& p, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  mla_tc_kernel<<<2 * p.workers, kThreads, kSmemBytes, stream>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace mla
