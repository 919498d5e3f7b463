// mla_simt.cu -- CUDA-core paged MLA kernel (16 heads per CTA, fp32 FMA).
//
// A plain, obviously-correct CUDA implementation of the same partition as the
// tensor-core kernel: worker w = blockIdx.x walks its tile range; blockIdx.y picks
// 16 query heads.  It gathers each 64-key tile of ckv|kpe rows into shared memory
// through kv_indices, scores it, runs the online softmax (running max, rescale,
// running sum: Modular MAX "mla_decoding_single_batch", "Flash attention v2
// algorithm") and accumulates o += p * ckv (V is the latent itself).
#include "common.cuh"
#include "launch.h"

namespace mla {

constexpr int kSimtHeads = 16;
constexpr int kSimtThreads = 256;
constexpr int kKeyWords = 289;  // 576 bf16 = 288 words, +1 word so key rows hit different banks

struct SimtShared {
  float q[kSimtHeads][kDimCkv + kDimKpe];
  uint32_t k[kTileKeys][kKeyWords];
  float p[kSimtHeads][kTileKeys];
  Cursor cur;
  long long T;
};

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(h);
}

__global__ void __launch_bounds__(kSimtThreads) mla_simt_kernel(MlaParams prm) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtShared& sh = *reinterpret_cast<SimtShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int w = blockIdx.x;
  const int h0 = blockIdx.y * kSimtHeads;
  const int hl = tid / 16;   // local head
  const int j = tid % 16;    // lane within the head's 16-thread group
  const int h = h0 + hl;

  PlanArgs pa{prm.kv_indptr, prm.qo_indptr, prm.batch, prm.num_kv_indices};
  if (tid < 32) {
    Cursor c;
    long long T = warp_plan(pa, w, prm.workers, &c);
    if (tid == 0) {
      sh.cur = c;
      sh.T = T;
    }
    if (w == 0 && blockIdx.y == 0) warp_write_empty_rows(prm);
  }
  __syncthreads();
  const long long T = sh.T;
  Walker walk;
  walk.init(pa, sh.cur, T, w, prm.workers);

  Segment seg;
  bool have_first = false;
  Segment first_seg{};
  while (walk.next(seg)) {
    if (seg.first) {
      have_first = true;
      first_seg = seg;
    }
    __syncthreads();
    for (int idx = tid; idx < kSimtHeads * (kDimCkv + kDimKpe); idx += kSimtThreads) {
      int hh = idx / (kDimCkv + kDimKpe), d = idx % (kDimCkv + kDimKpe);
      float v = 0.f;
      if (h0 + hh < prm.heads) {
        size_t rh = (size_t)seg.row * prm.heads + h0 + hh;
        v = d < kDimCkv ? __bfloat162float(prm.q_nope[rh * kDimCkv + d])
                        : __bfloat162float(prm.q_pe[rh * kDimKpe + d - kDimCkv]);
      }
      sh.q[hh][d] = v;
    }
    float m = -INFINITY, l = 0.f;
    float o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = 0.f;

    for (int tile = seg.t_begin; tile < seg.t_end; ++tile) {
      const int key0 = tile * kTileKeys;
      const int nvalid = min(kTileKeys, seg.len - key0);
      __syncthreads();
      // Gather 64 key rows (1152 B each: 64 x 16 B of ckv, 8 x 16 B of kpe).
      for (int v = tid; v < kTileKeys * 72; v += kSimtThreads) {
        int r = v / 72, c = v % 72;
        uint4 vec = make_uint4(0, 0, 0, 0);
        if (r < nvalid) {
          int slot = __ldg(prm.kv_indices + seg.kv0 + key0 + r);
          if (slot >= 0 && slot < prm.num_slots) {
            const uint4* src = c < 64
                ? reinterpret_cast<const uint4*>(prm.ckv + (size_t)slot * kDimCkv) + c
                : reinterpret_cast<const uint4*>(prm.kpe + (size_t)slot * kDimKpe) + (c - 64);
            vec = __ldg(src);
          }
        }
        uint32_t* dst = &sh.k[r][c * 4];
        dst[0] = vec.x; dst[1] = vec.y; dst[2] = vec.z; dst[3] = vec.w;
      }
      __syncthreads();
      float s[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int key = j + 16 * kk;
        float acc = 0.f;
        const float* q = sh.q[hl];
        const uint32_t* kr = sh.k[key];
#pragma unroll 8
        for (int wd = 0; wd < 288; ++wd) {
          float2 kv = bf2_to_f2(kr[wd]);
          acc = fmaf(q[2 * wd], kv.x, acc);
          acc = fmaf(q[2 * wd + 1], kv.y, acc);
        }
        s[kk] = key < nvalid ? acc * prm.scale_log2 : -INFINITY;
      }
      float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m, mx);
      const float alpha = fast_exp2(m - m_new);  // m = -inf on the first tile -> 0
      float ps = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float pv = fast_exp2(s[kk] - m_new);
        sh.p[hl][j + 16 * kk] = pv;
        ps += pv;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l = l * alpha + ps;
      m = m_new;
#pragma unroll
      for (int k = 0; k < 32; ++k) o[k] *= alpha;
      __syncthreads();
      for (int key = 0; key < nvalid; ++key) {
        const float pv = sh.p[hl][key];
        const uint32_t* vr = sh.k[key];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float2 v2 = bf2_to_f2(vr[j + 16 * k]);
          o[2 * k] = fmaf(pv, v2.x, o[2 * k]);
          o[2 * k + 1] = fmaf(pv, v2.y, o[2 * k + 1]);
        }
      }
    }
    // Epilogue: thread (hl, j) owns dims 2q, 2q+1 for q = j + 16k.
    if (h < prm.heads) {
      const float inv_l = 1.f / l;
      const float lse2 = m + fast_log2(l);
      if (seg.whole) {
        __nv_bfloat16* dst = prm.out + ((size_t)seg.row * prm.heads + h) * kDimCkv;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int q = j + 16 * k;
          *reinterpret_cast<__nv_bfloat162*>(dst + 2 * q) =
              __floats2bfloat162_rn(o[2 * k] * inv_l, o[2 * k + 1] * inv_l);
        }
        if (j == 0) prm.lse[(size_t)seg.row * prm.heads + h] = lse2 * 0.69314718055994531f;
      } else {
        const size_t frag = ((size_t)w * 2 + seg.slot) * prm.heads + h;
        float* dst = prm.part_o + frag * kDimCkv;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int q = j + 16 * k;
          *reinterpret_cast<float2*>(dst + 2 * q) = make_float2(o[2 * k] * inv_l, o[2 * k + 1] * inv_l);
        }
        if (j == 0) prm.part_lse[frag] = lse2;
      }
    }
  }
  if (blockIdx.y == 0 && tid == 0) prm.records[w] = make_record(have_first, first_seg, T, prm.workers);
}

cudaError_t launch_simt(const MlaParams& p, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(mla_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(SimtShared));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid(p.workers, (p.heads + kSimtHeads - 1) / kSimtHeads);
  mla_simt_kernel<<<grid, kSimtThreads, sizeof(SimtShared), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
