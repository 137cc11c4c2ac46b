// Router keys on the tensor cores (T > 1).
//
// "Three workload shapes" section of the Lily pages: the router scores every
// expert for every token; the layer computes the scores in fp32.  The bf16
// token row times the fp32 router row is evaluated as three bf16 GEMMs:
// router = hi + mid + lo with hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid) (each subtraction exact in fp32, the three parts
// carry 24 significant bits), and every bf16 x bf16 product is exact in fp32,
// so key = sum_k x_k*hi_k + x_k*mid_k + x_k*lo_k accumulated in fp32 differs
// from the fp32 dot product only by summation order.
//
//   router_split_kernel  fp32 [E][H] -> bf16 [3][E][H] (hi, mid, lo); run once
//                        per set of weights (moe_router_split) or, when the
//                        caller passes no split, inside the call
//   router_tc_kernel     D[e][t] = sum over parts of A_p[e] . x[t] (tcgen05,
//                        A and B from shared memory, fp32 accumulate in
//                        tensor memory), keys[t][e] = D + bias[e]
// One work item = 128 experts x N tokens (N = 32/64/128 by T) x one of KS
// slices of K (KS chosen so that the items fill the SMs; with KS > 1 each
// item writes fp32 partial sums and the top-k kernel adds the KS slices in
// order before it selects, so the keys do not depend on timing); warp 0 issues
// TMA (three 128x64 A boxes + one N x 64 B box per k-block, 128B swizzle),
// warp 1 issues the MMAs, warps 4-7 drain the accumulator.  Waits are bounded
// as in the expert kernels.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int RM = 128;       // experts per item
constexpr int RKB = 64;       // K per stage
constexpr int RSTAGES = 3;
constexpr int RTHREADS = 256;
constexpr int A_PART = RM * 128;  // one 128-row x 128-byte box
constexpr int B_MAX = 128 * 128;
constexpr int R_STAGE = 3 * A_PART + B_MAX;
constexpr int R_SMEM = RSTAGES * R_STAGE + 1024 + 1024;
constexpr unsigned long long R_TIMEOUT_NS = 1000000000ull;

struct RArgs {
  float *keys;     // [T][E] keys, or with KS > 1 the partial sums [KS][T][E]
  const float *bias;  // added when KS == 1 (else by the top-k kernel, after the slices)
  int32_t *status;
  int T, E, H, N, KS;
  int32_t *zero;  // nzero ints set to 0 (the top-k's histograms), or null
  int nzero;
};

struct RMisc {
  uint64_t full[RSTAGES], empty[RSTAGES];
  uint64_t acc_full, acc_empty, final_bar;
  uint32_t tmem;
  int abort_flag;
};

__device__ __forceinline__ bool rwait(uint64_t *bar, uint32_t parity, RMisc *m, int32_t *status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  uint32_t n = 0;
  while (!ptx::mbar_try_wait(bar, parity)) {
    if ((++n & 31u) == 0) {
      if (*reinterpret_cast<volatile int *>(&m->abort_flag)) return false;
      if (ptx::globaltimer() - t0 > R_TIMEOUT_NS) {
        *reinterpret_cast<volatile int *>(&m->abort_flag) = 1;
        set_status(status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ void rdrain(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > R_TIMEOUT_NS) return;
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void router_split_kernel(const float4 *__restrict__ w, size_t n4, uint2 *__restrict__ hi,
                                    uint2 *__restrict__ mid, uint2 *__restrict__ lo) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = w[i];
  const float x[4] = {v.x, v.y, v.z, v.w};
  uint16_t h[4], md[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat16 bh = __float2bfloat16_rn(x[j]);
    const float r1 = x[j] - __bfloat162float(bh);
    const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(bm);
    h[j] = __bfloat16_as_ushort(bh);
    md[j] = __bfloat16_as_ushort(bm);
    l[j] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
  }
  hi[i] = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
  mid[i] = make_uint2(md[0] | ((uint32_t)md[1] << 16), md[2] | ((uint32_t)md[3] << 16));
  lo[i] = make_uint2(l[0] | ((uint32_t)l[1] << 16), l[2] | ((uint32_t)l[3] << 16));
}

__global__ void __launch_bounds__(RTHREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                     const RArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // offset the shared pointer itself (not an integer cast), so accesses stay
  // shared-memory loads rather than generic ones
  uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  RMisc *m = reinterpret_cast<RMisc *>(smem + RSTAGES * R_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 3) {
    ptx::tmem_alloc(&m->tmem, 128);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < RSTAGES; ++i) {
      ptx::mbar_init(&m->full[i], 1);
      ptx::mbar_init(&m->empty[i], 1);
    }
    ptx::mbar_init(&m->acc_full, 1);
    ptx::mbar_init(&m->acc_empty, 128);
    ptx::mbar_init(&m->final_bar, 1);
    m->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // launched as a programmatic dependent of the kernel before it (which may
  // write x): everything above overlapped its tail, nothing below does
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = blockIdx.x * RTHREADS + threadIdx.x; i < a.nzero; i += gridDim.x * RTHREADS) a.zero[i] = 0;
  const uint32_t tmem = m->tmem;
  const int MT = a.E / RM;
  const int n_items = ((a.T + a.N - 1) / a.N) * MT * a.KS;
  const int KB = a.H / RKB / a.KS;  // k-blocks of one slice
  const uint32_t b_bytes = (uint32_t)a.N * 128u;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tma);
      ptx::prefetch_tmap(&tmb);
      uint32_t c = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int ks = item % a.KS, ti = item / a.KS, tt = ti / MT, et = ti - tt * MT;
        for (int kb = 0; kb < KB; ++kb, ++c) {
          const int s = c % RSTAGES;
          if (!rwait(&m->empty[s], ((c / RSTAGES) & 1u) ^ 1u, m, a.status)) {
            ok = false;
            break;
          }
          uint8_t *st = smem + s * R_STAGE;
          const int k0 = (ks * KB + kb) * RKB;
          ptx::mbar_arrive_expect_tx(&m->full[s], 3u * A_PART + b_bytes);
          for (int p = 0; p < 3; ++p)
            ptx::tma_load_2d(st + p * A_PART, &tma, &m->full[s], k0, p * a.E + et * RM);
          ptx::tma_load_2d(st + 3 * A_PART, &tmb, &m->full[s], k0, tt * a.N);
        }
      }
      if (!ok) {
        const uint32_t n = c < (uint32_t)RSTAGES ? c : (uint32_t)RSTAGES;
        for (uint32_t i = 1; i <= n; ++i) rdrain(&m->full[(c - i) % RSTAGES], ((c - i) / RSTAGES) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32((uint32_t)a.N);
      uint32_t c = 0, itc = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        if (!rwait(&m->acc_empty, (itc & 1u) ^ 1u, m, a.status)) break;
        ptx::tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++c) {
          const int s = c % RSTAGES;
          if (!rwait(&m->full[s], (c / RSTAGES) & 1u, m, a.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t base = ptx::smem_u32(smem + s * R_STAGE);
#pragma unroll
          for (int p = 0; p < 3; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma_ss(tmem, ptx::sdesc_sw128(base + p * A_PART + 32 * i),
                     ptx::sdesc_sw128(base + 3 * A_PART + 32 * i), idesc, (uint32_t)(kb | p | i));
          ptx::mma_commit(&m->empty[s]);
        }
        if (!ok) break;
        ptx::mma_commit(&m->acc_full);
        ++itc;
      }
      ptx::mma_commit(&m->final_bar);
      rdrain(&m->final_bar, 0);
    }
  } else if (warp >= 4) {
    const int q = warp & 3;
    const int e_local = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t itc = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int ks = item % a.KS, ti = item / a.KS, tt = ti / MT, et = ti - tt * MT;
      if (!__all_sync(0xffffffffu, rwait(&m->acc_full, itc & 1u, m, a.status))) break;
      ptx::tc_fence_after();
      const int e = et * RM + e_local;
      const float b = (a.bias && a.KS == 1) ? a.bias[e] : 0.f;
      float *out = a.keys + (size_t)ks * a.T * a.E;
      for (int ch = 0; ch < a.N / 16; ++ch) {
        uint32_t v[16];
        ptx::tmem_ld_x16(tmem + lane_base + ch * 16, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = tt * a.N + ch * 16 + i;
          if (t < a.T) out[(size_t)t * a.E + e] = __uint_as_float(v[i]) + b;
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&m->acc_empty);
      ++itc;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 128);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

// bf16 [rows][cols] tensor, boxes of box_rows x 64 elements, 128B swizzle.
cudaError_t bf16_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorInitializationError;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool router_tc_supported(int E, int H) { return E % RM == 0 && H % RKB == 0; }

namespace {
int router_n(int T) { return T >= 2048 ? 128 : (T >= 512 ? 64 : 32); }
}  // namespace

int router_tc_slices(int T, int E, int H, int num_sms) {
  const int items = ((T + router_n(T) - 1) / router_n(T)) * (E / RM), kb = H / RKB;
  int ks = 1;
  while (ks < 8 && items * ks * 2 <= num_sms && kb % (ks * 2) == 0 && kb / (ks * 2) >= 4) ks *= 2;
  return ks;
}

size_t router_tc_partial_floats(int Tmax, int E, int H, int num_sms) {
  size_t most = 0;
  for (int T = 1; T <= Tmax; ++T) {
    const int ks = router_tc_slices(T, E, H, num_sms);
    if (ks > 1 && (size_t)ks * T > most) most = (size_t)ks * T;
  }
  return most * (size_t)E;
}

cudaError_t router_tc_prepare() {
  return cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM);
}

cudaError_t launch_router_split(const float *router, int E, int H, uint16_t *split, cudaStream_t s) {
  const size_t n = (size_t)E * H;
  router_split_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const float4 *>(router), n / 4, reinterpret_cast<uint2 *>(split),
      reinterpret_cast<uint2 *>(split + n), reinterpret_cast<uint2 *>(split + 2 * n));
  return cudaGetLastError();
}

cudaError_t launch_router_tc(const uint16_t *x, int T, int H, const float *router, int E, const float *bias,
                             const uint16_t *split_given, uint16_t *split, float *partial, float *keys,
                             int32_t *status, int32_t *zero, int nzero, int num_sms, int *ks_out, int *launches,
                             cudaStream_t s) {
  const bool pdl = prof_chain(MOE_KERNEL_ROUTER);  // a dependent of the kernel before it (not of the split)
  prof_before(MOE_KERNEL_ROUTER, s);
  cudaError_t e = cudaSuccess;
  if (split_given) {
    split = const_cast<uint16_t *>(split_given);
  } else {
    if ((e = launch_router_split(router, E, H, split, s)) != cudaSuccess) return e;
    ++*launches;
  }
  const int N = router_n(T), KS = router_tc_slices(T, E, H, num_sms);
  CUtensorMap ta, tb;
  if ((e = bf16_map(&ta, split, 3 * E, H, RM)) != cudaSuccess) return e;
  if ((e = bf16_map(&tb, x, T, H, N)) != cudaSuccess) return e;
  RArgs a{KS > 1 ? partial : keys, bias, status, T, E, H, N, KS, zero, zero ? nzero : 0};
  const int items = ((T + N - 1) / N) * (E / RM) * KS;
  e = launch_dep(pdl && split_given != nullptr, router_tc_kernel, dim3(items < num_sms ? items : num_sms),
                 dim3(RTHREADS), R_SMEM, s, ta, tb, a);
  prof_after(MOE_KERNEL_ROUTER, s);
  if (e != cudaSuccess) return e;
  ++*launches;
  *ks_out = KS;
  return cudaGetLastError();
}

}  // namespace moe
