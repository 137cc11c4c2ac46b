// Tensor-core grouped expert GEMMs (tcgen05, sm_103a).
//
// "Prefill" section of the Lily pages: the 4-bit groupwise-affine weights are
// rebuilt to bf16 tile by tile inside the grouped GEMM and accumulated in
// FP32, so no unpacked weight array reaches memory; the grouped GEMMs follow
// a device-built block map (one tile = up to 128 (gate/up) or 256 (down)
// rows of one expert).
//
// One persistent CTA per SM takes work items (block-map tile, 128 output
// features): the code producer draws the next item number from a queue (a
// global counter per GEMM, zeroed by the scatter kernel before every layer),
// so the SMs stay busy to the end whatever the tiles' sizes, and hands its
// block-map entry to the CTA's other roles through a ring in shared memory.  The packed weights are the MMA's A operand (M = 128 rows of
// output features) and the tile's token rows are B (N = rows rounded up to
// 16), so a weight tile is rebuilt once for all of an expert's tokens:
//   warp 0      TMA: packed 4-bit codes, 128 rows x 256 codes per box, 128B
//               swizzle, one box per matrix per stage of 4 k-blocks
//   warps 1, 3  one thread each issues tcgen05.mma (A from tensor memory, B
//               from shared memory, D fp32 in tensor memory) and commits;
//               warp 3 also allocates and frees the tensor memory
//   warp 2      TMA: the tile's token rows, contiguous in the source (x rows
//               gathered in perm order for the routed experts, x itself for
//               the shared expert, h for the down GEMM), 128B-swizzled
//   warps 4-15  three warpgroups: dequantise a k-block of every matrix (64
//               codes of a row -> 32 bf16x2, w = bf16_rne(scale*q + bias))
//               straight into tensor memory with tcgen05.st, then run the
//               epilogue: gate/up: h = bf16(silu(g) * u); down: y = bf16(acc)
// Tensor memory (512 columns), gate/up: D_gate [0,128), D_up [128,256), four
// A slots of 64 columns at 256 (gate at +0, up at +32; 32 columns = 64 bf16
// of K).  Down, one output tile per item (tiles of up to 192 rows): two
// accumulators D0 [0,192) and D1 [192,384), so that the MMA runs the next
// item while the epilogue drains the last one, and four A slots of 32
// columns at 384.  Down, two output tiles per item (tiles of up to 128 rows,
// the layout of gate/up): the two tiles share the item's token rows, which
// halves their reads where the tiles are short.  A k-block's token rows and
// its A slot form one slot of a four-slot ring.
// Every wait is bounded: after one second the kernel records
// MOE_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees tensor memory
// and exits.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;         // output features per work item (= TMEM lanes)
constexpr int KBLK = 64;        // k-block = one quantisation group
constexpr int STAGE_KB = 4;     // k-blocks per code stage (one TMA box per matrix)
constexpr int BOX = BM * 128;   // one TMA box: 128 rows x 128 bytes (256 codes)
constexpr int NSLOT = 4;        // k-block ring: A slots in tensor memory (64 columns each) + token-row slots
static_assert(STAGE_KB <= NSLOT, "an item's first code stage must fit the k-block ring (deferred epilogue)");
constexpr int NISS = 2;         // MMA-issuing threads (warps 1 and 3)
constexpr int NWG = 3;                    // dequant/epilogue warpgroups
constexpr int THREADS = 128 + NWG * 128;  // 4 role warps + the warpgroups
constexpr uint32_t TMEM_COLS = 512;
constexpr unsigned long long TIMEOUT_NS = 1000000000ull;

constexpr int SBOX = BM * 16;  // one scale (or bias) box: 128 rows x 8 groups of bf16

// Kernel modes: the gate/up GEMM (+ SwiGLU); the down GEMM with one
// 128-feature output tile per item; the down GEMM with two output tiles per
// item (features 256 m .. 256 m + 255), which share the item's token rows
// exactly as gate and up do; and the same with short tiles (at most
// TC_SHORT_ROWS rows), whose accumulators are small enough to keep two items
// in flight.
enum { MODE_DOWN = 0, MODE_GATEUP = 1, MODE_DOWN2 = 2, MODE_DOWN2_SHORT = 3 };

template <int MODE>
struct Cfg {
  // two weight tiles per k-block against the same token rows (gate and up,
  // or two output tiles of down), each with its own accumulator
  static constexpr bool TWO = MODE != MODE_DOWN;
  static constexpr int NMAT = TWO ? 2 : 1;
  // Token rows per work item (the MMA's N).  The accumulators (NMAT tiles x
  // NBUF items in flight, N columns each) sit next to the A slots in tensor
  // memory: N <= 128 with two tiles and one item, N <= 192 with one tile and
  // two items, N <= 64 with two tiles and two items.
  static constexpr int MAXN = MODE == MODE_DOWN2_SHORT ? TC_SHORT_ROWS : TWO ? 128 : TC_DOWN_ROWS;
  static constexpr int NBUF = (TWO && MODE != MODE_DOWN2_SHORT) ? 1 : 2;  // accumulators (items in flight)
  static constexpr int D_UP = MAXN;                      // second tile's accumulator, after the first
  static constexpr int D_BUF = NBUF == 2 ? NMAT * MAXN : 0;  // columns from one item's accumulators to the next
  static constexpr int A_COL = NBUF * NMAT * MAXN;       // first A slot
  static constexpr int A_SLOT = TWO ? 64 : 32;     // columns per A slot
  static_assert(A_COL + NSLOT * A_SLOT <= (int)TMEM_COLS, "tensor memory");
  static constexpr int B_SLOT = MAXN * 128;  // one k-block of MAXN token rows
  // Code stages (4 k-blocks each, from HBM) and the k-block ring (token rows
  // in shared memory + dequantised weights in tensor memory) share the
  // shared memory.
  static constexpr int CSTAGES = TWO ? 3 : 4;
  // per stage: codes of each matrix, then (scale, bias) boxes of each matrix
  static constexpr int STAGE_BYTES = NMAT * BOX + NMAT * 2 * SBOX;
  static constexpr int OFF_B = CSTAGES * STAGE_BYTES;
  // epilogue staging: per dequant warp two buffers of 16 rows x 32 features
  static constexpr int EPI_BUF = 16 * 32 * 2;
  static constexpr int OFF_EPI = OFF_B + NSLOT * B_SLOT;
  static constexpr int OFF_MISC = OFF_EPI + NWG * 4 * 2 * EPI_BUF;
  static constexpr int SMEM = OFF_MISC + 1024 /* misc */ + 1024 /* alignment slack */;
  static_assert(CSTAGES <= 8, "code_full / code_empty arrays");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Tensor maps: codes of matrix 0/1, and (when tma_scales) scale/bias of
// matrix 0/1 as [rows][K/64] bf16 with 128 x 8 boxes.
struct TcMaps {
  CUtensorMap code[2];
  CUtensorMap sc[2];
  CUtensorMap bi[2];
  // token rows: a bf16 tensor [rows][K] with 128B-swizzled boxes of one
  // k-block (64 values) x 128 / 64 / 32 / 16 rows: h (down) or the x rows
  // gathered in block-map row order (gate/up), both in the interleaved K order
  CUtensorMap act[4];
  // the output (h or y) as bf16 [rows][NOUT], boxes of 32 features x 16
  // rows, for the epilogue's TMA stores (one per warp and chunk)
  CUtensorMap out;
};

struct TcArgs {
  const int32_t *blockmap, *n_tiles;
  int32_t *item_counter;          // next item number, zero at launch; null: items round-robin
  const uint16_t *sc[2], *bi[2];  // scale / bias arrays of the matrices
  uint16_t *out;                  // h [rows][NOUT] or y [rows][NOUT]
  int32_t *status;
  int T, k, E, K, NOUT;           // K: reduction length; NOUT: output features per expert
  int tma_scales;                 // scales/biases staged by TMA (K % 512 == 0)
  // The block map's last `first` tiles (the shared expert's: with few tokens
  // per routed expert, the largest) are handed out before the others, so the
  // items that finish last are short ones.
  int first;
  // Optional wait accounting (tracing aid): per CTA, cycles each role spent
  // in its barrier waits and in total, at trace[cta * 32 + trace_base + i].
  uint64_t *trace;
  int trace_base;
};

// Slots of the wait accounting (see TcArgs::trace).
enum {
  TW_TMA_EMPTY, TW_MMA_ACC, TW_MMA_READY, TW_UNUSED3, TW_LOAD_FREE, TW_DQ_CODE, TW_DQ_FREE, TW_DQ_ACC,
  TW_TMA_TOTAL, TW_MMA_TOTAL, TW_LOAD_TOTAL, TW_DQ_TOTAL, TW_ITEMS, TW_N
};

// f() (a wait), with its clock64 cycles added to acc when on.
template <typename F>
__device__ __forceinline__ bool timed(bool on, unsigned long long &acc, F f) {
  if (!on) return f();
  const long long t0 = clock64();
  const bool r = f();
  acc += (unsigned long long)(clock64() - t0);
  return r;
}

// The k-block ring: slot s holds k-block kb (s = kb % NSLOT of the CTA's
// running k-block count) -- its token rows in shared memory and its
// dequantised weights in tensor memory.  ready[s] completes when both have
// landed (the TMA bytes plus one arrival per dequant thread of each matrix);
// free[s] when every MMA that read the slot has completed (one commit per
// issuer).
// Items in flight between the code producer and the other roles.
constexpr int IRING = 8;
// Consumers of an item-ring slot: the token loader, the MMA issuers and every
// dequant warp.
constexpr int ITEM_READERS = 1 + NISS + NWG * 4;

struct Misc {
  int4 item[IRING];  // (expert, first row, rows, m-tile); expert < 0: no more items
  uint64_t item_full[IRING], item_empty[IRING];
  uint64_t code_full[8], code_empty[8];
  uint64_t ready[NSLOT], free[NSLOT];
  uint64_t acc_full[2], acc_empty[2], final_bar;  // per accumulator
  uint32_t tmem;
  int abort_flag;
};

struct Item {
  int e, row0, nrows, n_mma, mt;
};

// Block-map entry of item number `item` (of n_tiles * MT) as a ring entry;
// items count from the map's last a.first tiles, then from its start.
template <int MAXN>
__device__ __forceinline__ int4 item_entry(const TcArgs &a, int item, int MT, int n_tiles) {
  const int t = item / MT;
  const int first = a.first < n_tiles ? a.first : n_tiles;
  const int tile = t < first ? n_tiles - first + t : t - first;
  const int4 ent = reinterpret_cast<const int4 *>(a.blockmap)[tile];
  return make_int4(ent.x, ent.y, min(ent.z, MAXN), item - t * MT);
}

__device__ __forceinline__ Item as_item(int4 ent) {
  Item it;
  it.e = ent.x;
  it.row0 = ent.y;
  it.nrows = ent.z;
  it.mt = ent.w;
  it.n_mma = max(16, (it.nrows + 15) & ~15);
  return it;
}

// Bounded wait on an mbarrier phase; false (and the CTA-wide abort flag) on
// timeout or when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Misc *m, int32_t *status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  uint32_t n = 0;
  while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u)) {
    if ((++n & 7u) == 0) {
      if (*reinterpret_cast<volatile int *>(&m->abort_flag)) return false;
      if (ptx::globaltimer() - t0 > TIMEOUT_NS) {
        *reinterpret_cast<volatile int *>(&m->abort_flag) = 1;
        set_status(status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > TIMEOUT_NS) return;
}

// The n-th item of this CTA from the ring (all lanes of the calling warp, or
// one thread with warp_wide false); false on a failed wait.
__device__ __forceinline__ bool read_item(Misc *m, uint32_t n, int4 &ent, int32_t *status, bool warp_wide) {
  const int s = n % IRING;
  const bool got = wait_bar(&m->item_full[s], (n / IRING) & 1u, m, status);
  if (warp_wide ? !__all_sync(0xffffffffu, got) : !got) return false;
  const volatile int *src = reinterpret_cast<volatile int *>(&m->item[s]);
  ent = make_int4(src[0], src[1], src[2], src[3]);
  if (warp_wide) __syncwarp();
  if (!warp_wide || (threadIdx.x & 31) == 0) ptx::mbar_arrive(&m->item_empty[s]);
  return true;
}

// K order inside the tensor-core GEMMs.  Within every run of 8 values along
// K the operands are stored as (0,4), (1,5), (2,6), (3,7) pairs: a packed code
// word holds code i at bits 4i, so the pair (j, j+4) sits at bits 4j and
// 4j+16 and comes out with one shift and one and-or, and the token rows (x
// gathered, h written by the gate/up epilogue) are stored in the same order,
// so the MMA sums exactly the same products.
//   ilv_pos(f): storage position of value f of a run.
__device__ __forceinline__ int ilv_pos(int f) { return (f & ~7) | ((f & 3) << 1) | ((f >> 2) & 1); }

// The bf16 values of groups g0 .. g0+n-1 of one row (n <= 4), packed two
// per 32-bit word (group g0 in the low half of .x).
__device__ __forceinline__ uint2 load_groups(const uint16_t *p, int n, bool vec) {
  if (vec && n == 4) return __ldg(reinterpret_cast<const uint2 *>(p));
  uint16_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = (i < n) ? __ldg(p + i) : 0;
  return make_uint2(v[0] | ((uint32_t)v[1] << 16), v[2] | ((uint32_t)v[3] << 16));
}

// bf16x2 with group j's value (of a load_groups word pair) in both halves.
__device__ __forceinline__ __nv_bfloat162 pick_group(uint2 g, int j) {
  const uint32_t w = (j & 2) ? g.y : g.x;
  const uint32_t h = (j & 1) ? (w >> 16) : (w & 0xFFFFu);
  const uint32_t u = h | (h << 16);
  return *reinterpret_cast<const __nv_bfloat162 *>(&u);
}

__device__ __forceinline__ void trace_put(const TcArgs &a, int slot, unsigned long long v) {
  if (a.trace && blockIdx.x < MOE_TRACE_CTAS) a.trace[blockIdx.x * MOE_TRACE_SLOTS + a.trace_base + slot] = v;
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    experts_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
  using C = Cfg<MODE>;
  constexpr bool GATEUP = MODE == MODE_GATEUP, PAIR = MODE == MODE_DOWN2 || MODE == MODE_DOWN2_SHORT;
  // first weight row of matrix mat of an item: its output tile (two per item
  // when PAIR)
  auto w_row = [&](const Item &it, int mat) {
    return it.e * a.NOUT + (PAIR ? (2 * it.mt + mat) : it.mt) * BM;
  };
  extern __shared__ uint8_t smem_raw[];
  // offset the shared pointer itself (not an integer cast), so accesses stay
  // shared-memory loads rather than generic ones
  uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc *m = reinterpret_cast<Misc *>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 3) {
    ptx::tmem_alloc(&m->tmem, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < IRING; ++i) {
      ptx::mbar_init(&m->item_full[i], 1);
      ptx::mbar_init(&m->item_empty[i], ITEM_READERS);
    }
    for (int i = 0; i < C::CSTAGES; ++i) {
      ptx::mbar_init(&m->code_full[i], 1);
      ptx::mbar_init(&m->code_empty[i], NWG * 4);
    }
    for (int i = 0; i < NSLOT; ++i) {
      ptx::mbar_init(&m->ready[i], 1 + 128);  // token-row TMA + the warpgroup that rebuilt the k-block
      ptx::mbar_init(&m->free[i], NISS);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&m->acc_full[b], NISS);
      ptx::mbar_init(&m->acc_empty[b], NWG * 128);
    }
    ptx::mbar_init(&m->final_bar, NISS);
    m->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = m->tmem;

  const int MT = a.NOUT / (PAIR ? 2 * BM : BM);  // items per block-map tile
  const int KB = a.K / KBLK;  // a multiple of NSLOT (K % 256 == 0)
  const int NST = (KB + STAGE_KB - 1) / STAGE_KB;
  const int n_tiles = *a.n_tiles;
  const int n_items = n_tiles * MT;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (codes, scales)
    if (lane == 0) {
      const bool tr = a.trace != nullptr;
      const long long t_start = clock64();
      unsigned long long w_empty = 0;
      for (int mat = 0; mat < C::NMAT; ++mat) {
        ptx::prefetch_tmap(&maps.code[mat]);
        if (a.tma_scales) {
          ptx::prefetch_tmap(&maps.sc[mat]);
          ptx::prefetch_tmap(&maps.bi[mat]);
        }
      }
      uint32_t cs = 0;
      bool ok = true;
      // Items are drawn from the queue two ahead of the one being loaded, so
      // the counter's and the block map's round trips overlap earlier work:
      // nxt = the next item's entry, idx2 = the number after it.
      // With a.item_counter null the items go round-robin instead (item
      // number blockIdx.x + n * gridDim.x).
      int stat = blockIdx.x;
      auto draw = [&]() {
        if (a.item_counter) return atomicAdd(a.item_counter, 1);
        const int i = stat;
        stat += gridDim.x;
        return i;
      };
      int idx2 = draw();
      int4 nxt = idx2 < n_items ? item_entry<C::MAXN>(a, idx2, MT, n_tiles) : make_int4(-1, 0, 0, 0);
      idx2 = nxt.x < 0 ? n_items : draw();
      for (uint32_t n = 0; ok; ++n) {
        // the next item, posted to the ring before its codes
        const int s = n % IRING;
        if (!wait_bar(&m->item_empty[s], ((n / IRING) & 1u) ^ 1u, m, a.status)) break;
        const int4 ent = nxt;
        m->item[s] = ent;
        ptx::mbar_arrive(&m->item_full[s]);
        if (ent.x < 0) break;
        nxt = idx2 < n_items ? item_entry<C::MAXN>(a, idx2, MT, n_tiles) : make_int4(-1, 0, 0, 0);
        if (nxt.x >= 0) idx2 = draw();
        const Item it = as_item(ent);
        for (int st = 0; st < NST; ++st, ++cs) {
          const int slot = cs % C::CSTAGES;
          const uint32_t ph = (cs / C::CSTAGES) & 1u;
          if (!timed(tr, w_empty, [&] { return wait_bar(&m->code_empty[slot], ph ^ 1u, m, a.status); })) {
            ok = false;
            break;
          }
          const int kb0 = st * STAGE_KB;
          const uint32_t bytes = C::NMAT * (BOX + (a.tma_scales ? 2 * SBOX : 0));
          ptx::mbar_arrive_expect_tx(&m->code_full[slot], bytes);
          uint8_t *stage = smem + slot * C::STAGE_BYTES;
          for (int mat = 0; mat < C::NMAT; ++mat) {
            const int row_base = w_row(it, mat);
            ptx::tma_load_2d(stage + mat * BOX, &maps.code[mat], &m->code_full[slot], kb0 * (KBLK / 2), row_base);
            if (a.tma_scales) {  // the 8 groups around this stage's 4 (16-byte aligned boxes)
              uint8_t *sb = stage + C::NMAT * BOX + mat * 2 * SBOX;
              ptx::tma_load_2d(sb, &maps.sc[mat], &m->code_full[slot], kb0 & ~7, row_base);
              ptx::tma_load_2d(sb + SBOX, &maps.bi[mat], &m->code_full[slot], kb0 & ~7, row_base);
            }
          }
        }
      }
      if (!ok) {  // loads of the last stages may still be in flight
        const uint32_t n = cs < (uint32_t)C::CSTAGES ? cs : (uint32_t)C::CSTAGES;
        for (uint32_t i = 1; i <= n; ++i) {
          const uint32_t c = cs - i;
          drain_wait(&m->code_full[c % C::CSTAGES], (c / C::CSTAGES) & 1u);
        }
      }
      trace_put(a, TW_TMA_EMPTY, w_empty);
      trace_put(a, TW_TMA_TOTAL, (unsigned long long)(clock64() - t_start));
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // A thread issues at most one tcgen05.mma every ~50 cycles and every
    // instruction between them adds to that, so two threads issue, from a
    // loop unrolled over the ring's slots (constant addresses).  Each
    // accumulator column stays with one issuer, in K order, so the result
    // does not depend on how the two interleave: gate/up split by matrix,
    // down by halves of the tile's N.
    if (lane == 0) {
      const int iss = warp == 3 ? 1 : 0;
      const bool tr = a.trace != nullptr && iss == 0;
      const long long t_start = clock64();
      unsigned long long w_acc = 0, w_ready = 0;
      // descriptor of B slot 0 (128B-swizzled K-major); other slots and K
      // steps only move the address field in its low word
      const uint64_t bdesc0 = ptx::sdesc_sw128(ptx::smem_u32(smem + C::OFF_B));
      const uint32_t b_lo0 = (uint32_t)bdesc0, b_hi = (uint32_t)(bdesc0 >> 32);
      const int mat = C::TWO ? iss : 0;
      const uint32_t a_col = tmem + C::A_COL + (uint32_t)(mat * 32);
      uint32_t kbc = 0, itc = 0;
      bool ok = true;
      for (;;) {
        int4 ent;
        if (!read_item(m, itc, ent, a.status, false)) break;
        if (ent.x < 0) break;
        const Item it = as_item(ent);
        // this issuer's token columns [c0, c0 + nc)
        int c0 = 0, nc = it.n_mma;
        if (!C::TWO) {
          const int half = ((it.n_mma >> 1) + 15) & ~15;
          c0 = iss ? half : 0;
          nc = iss ? it.n_mma - half : half;
        }
        const uint32_t idesc = ptx::idesc_bf16_f32((uint32_t)(nc > 0 ? nc : 16));
        // accumulator itc % NBUF; its previous item's epilogue must have read it
        const uint32_t buf = itc % C::NBUF, use = itc / C::NBUF;
        const uint32_t d = tmem + buf * C::D_BUF + (uint32_t)(mat * C::D_UP + c0);
        const uint32_t b_lo = b_lo0 + (uint32_t)c0 * 8u;  // c0 rows of 128 B, in 16-byte units
        if (!timed(tr, w_acc, [&] { return wait_bar(&m->acc_empty[buf], (use & 1u) ^ 1u, m, a.status); })) break;
        ptx::tc_fence_after();
        for (int kb = 0; kb < KB && ok; kb += NSLOT, kbc += NSLOT) {
          const uint32_t ph = (kbc / NSLOT) & 1u;
#pragma unroll
          for (int j = 0; j < NSLOT; ++j) {
            if (!timed(tr, w_ready, [&] { return wait_bar(&m->ready[j], ph, m, a.status); })) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            if (nc > 0)
              ptx::mma_ts_kblock(d, a_col + j * C::A_SLOT, b_lo + (uint32_t)(j * (C::B_SLOT >> 4)), b_hi, idesc,
                                 (uint32_t)(kb + j));
            ptx::mma_commit(&m->free[j]);
          }
        }
        if (!ok) break;
        ptx::mma_commit(&m->acc_full[buf]);
        ++itc;
      }
      // every MMA this thread issued has completed before tensor memory is freed
      ptx::mma_commit(&m->final_bar);
      drain_wait(&m->final_bar, 0);
      trace_put(a, TW_MMA_ACC, w_acc);
      trace_put(a, TW_MMA_READY, w_ready);
      trace_put(a, TW_MMA_TOTAL, (unsigned long long)(clock64() - t_start));
      trace_put(a, TW_ITEMS, itc);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ token-row TMA
    // (Launched as a programmatic dependent, the kernel may start while the
    // kernel before it -- the gather of x, or gate/up for down -- still runs:
    // the weights' copies and every other role go ahead, and only the token
    // rows, that kernel's output, wait for it to finish.)
    // The rows of a tile are contiguous (down: routed rows of h in perm order,
    // then the shared expert's; gate/up: the x rows gathered in the same
    // order), so each k-block of the
    // tile's n_mma rows arrives in a few TMA boxes (128 rows at a time, then
    // 64 / 32 / 16), already in the MMA's 128B-swizzled K-major layout.  Rows
    // past the tile belong to the next tile (or lie past the tensor and read
    // as zero): they only feed MMA columns the epilogue never stores.
    if (lane == 0) {
      const bool tr = a.trace != nullptr;
      const long long t_start = clock64();
      unsigned long long w_free = 0;
      for (int i = 0; i < 4; ++i) ptx::prefetch_tmap(&maps.act[i]);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      uint32_t kbc = 0;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n) {
        int4 ent;
        if (!read_item(m, n, ent, a.status, false) || ent.x < 0) break;
        const Item it = as_item(ent);
        const CUtensorMap *mp = maps.act;
        const int rb = it.row0;
        for (int kb = 0; kb < KB; ++kb, ++kbc) {
          const int slot = kbc % NSLOT;
          if (!timed(tr, w_free, [&] { return wait_bar(&m->free[slot], ((kbc / NSLOT) & 1u) ^ 1u, m, a.status); })) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&m->ready[slot], (uint32_t)it.n_mma * 128u);
          uint8_t *bs = smem + C::OFF_B + slot * C::B_SLOT;
          int r = 0;
          for (; it.n_mma - r >= 128; r += 128)
            ptx::tma_load_2d(bs + r * 128, &mp[0], &m->ready[slot], kb * KBLK, rb + r);
#pragma unroll
          for (int i = 1; i < 4; ++i) {
            const int h = 128 >> i;
            if (it.n_mma - r >= h) {
              ptx::tma_load_2d(bs + r * 128, &mp[i], &m->ready[slot], kb * KBLK, rb + r);
              r += h;
            }
          }
        }
      }
      if (!ok) {  // the last slots' loads may still be in flight
        const uint32_t n = kbc < (uint32_t)NSLOT ? kbc : (uint32_t)NSLOT;
        for (uint32_t i = 1; i <= n; ++i) {
          const uint32_t c = kbc - i;
          drain_wait(&m->ready[c % NSLOT], (c / NSLOT) & 1u);
        }
      }
      trace_put(a, TW_LOAD_FREE, w_free);
      trace_put(a, TW_LOAD_TOTAL, (unsigned long long)(clock64() - t_start));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dequant + epilogue
    // Work unit = one k-block of every matrix (gate and up, or down): the
    // CTA's running k-block kbg goes to warpgroup kbg % NWG, which rebuilds
    // it into A slot kbg % NSLOT and arrives once on that slot's ready
    // barrier; epilogue chunks of 16 columns are dealt round-robin.
    // A slot's free barrier is waited on by phase parity, which is exact only
    // while the waiter is at most one phase ahead of the slot.  That holds
    // here: a warpgroup's consecutive k-blocks are NWG <= NSLOT apart, so its
    // previous wait already saw the MMA past k-block kbg - 2 NSLOT, and every
    // warp meets the MMA at the end of each item (acc_full) before it starts
    // the next.  A different unit order, or an epilogue moved past the next
    // item's first units, must keep this.
    const int wg = (warp - 4) >> 2, q = warp & 3;
    const int row = q * 32 + lane;  // weight row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int groups = a.K / KBLK;
    const bool vec = (groups % 4) == 0;
    const bool tr = a.trace != nullptr && warp == 4 && lane == 0;
    const long long t_start = clock64();
    unsigned long long w_code = 0, w_free = 0, w_acc = 0;
    uint32_t cs = 0, kbc = 0, itc = 0;
    bool ok = true;
    // (without scale boxes) the scales and biases of the next stage of the
    // item are loaded one stage ahead
    uint2 nsv[C::NMAT], nbv[C::NMAT];
    auto prefetch = [&](const Item &pi, int pst) {
      const int kb0 = pst * STAGE_KB, nkb = min(STAGE_KB, KB - kb0);
#pragma unroll
      for (int mt = 0; mt < C::NMAT; ++mt) {
        const size_t grow = (size_t)w_row(pi, mt) + row;
        nsv[mt] = load_groups(a.sc[mt] + grow * groups + kb0, nkb, vec);
        nbv[mt] = load_groups(a.bi[mt] + grow * groups + kb0, nkb, vec);
      }
    };
    // The epilogue of item number ic (this CTA's count): chunks of 16 token
    // columns dealt round-robin to the warpgroups, out of accumulator ic % NBUF.
    uint32_t epi_n = 0;  // whole chunks this warpgroup has stored by TMA
    auto epilogue = [&](const Item &ei, uint32_t ic) -> bool {
      const uint32_t buf = ic % C::NBUF, use = ic / C::NBUF;
      if (!__all_sync(0xffffffffu,
                      timed(tr, w_acc, [&] { return wait_bar(&m->acc_full[buf], use & 1u, m, a.status); }))) {
        ok = false;
        return false;
      }
      ptx::tc_fence_after();
      const uint32_t dcol = tmem + lane_base + buf * C::D_BUF;
      // gate/up writes h in the interleaved K order of the down GEMM (a
      // permutation within runs of 8, so within this warp's 32 features)
      const int pos = GATEUP ? ilv_pos(row) : row;
      // 16 token rows x this warp's 32 features of output tile `tile`
      auto put = [&](const uint16_t (&o)[16], int ch, int tile) {
        if (ch * 16 + 16 <= ei.nrows) {
          // a whole chunk: through this warp's staging buffer and one TMA
          // store of 16 rows x its 32 features (the buffer used two stores
          // ago must have been read by its store first)
          uint16_t *sb = reinterpret_cast<uint16_t *>(smem + C::OFF_EPI + ((warp - 4) * 2 + (epi_n & 1)) * C::EPI_BUF);
          if (lane == 0) ptx::bulk_wait_read<1>();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 16; ++i) sb[i * 32 + (pos & 31)] = o[i];
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&maps.out, sb, tile * BM + q * 32, ei.row0 + ch * 16);
            ptx::bulk_commit();
          }
          ++epi_n;
        } else {  // the tile's ragged last chunk: rows past it belong to the next tile
          uint16_t *orow = a.out + (size_t)ei.row0 * a.NOUT + (size_t)tile * BM + pos;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (ch * 16 + i < ei.nrows) orow[(size_t)(ch * 16 + i) * a.NOUT] = o[i];
        }
      };
      for (int ch = wg; ch < ei.n_mma / 16; ch += NWG) {
        uint32_t g[16], u[16];
        ptx::tmem_ld_x16(dcol + ch * 16, g);
        if (C::TWO) ptx::tmem_ld_x16(dcol + C::D_UP + ch * 16, u);
        ptx::tmem_wait_ld();
        uint16_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = f32_to_bf16(GATEUP ? silu(__uint_as_float(g[i])) * __uint_as_float(u[i]) : __uint_as_float(g[i]));
        put(o, ch, PAIR ? 2 * ei.mt : ei.mt);
        if (PAIR) {  // the item's second output tile
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = f32_to_bf16(__uint_as_float(u[i]));
          put(o, ch, 2 * ei.mt + 1);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&m->acc_empty[buf]);
      return true;
    };
    Item prev{0, 0, 0, 16, 0};
    bool has_prev = false;
    for (;;) {
      int4 ent;
      if (!read_item(m, itc, ent, a.status, true)) {
        ok = false;
        break;
      }
      if (ent.x < 0) break;
      const Item it = as_item(ent);
      if (!a.tma_scales) prefetch(it, 0);
      for (int st = 0; st < NST; ++st, ++cs) {
        const int kb0 = st * STAGE_KB, nkb = min(STAGE_KB, KB - kb0);
        uint2 sv[C::NMAT], bv[C::NMAT];
#pragma unroll
        for (int mt = 0; mt < C::NMAT; ++mt) {
          sv[mt] = nsv[mt];
          bv[mt] = nbv[mt];
        }
        if (!a.tma_scales && st + 1 < NST) prefetch(it, st + 1);
        const int cslot = cs % C::CSTAGES;
        if (!__all_sync(0xffffffffu, timed(tr, w_code, [&] {
              return wait_bar(&m->code_full[cslot], (cs / C::CSTAGES) & 1u, m, a.status);
            }))) {
          ok = false;
          break;
        }
        if (a.tma_scales) {  // this row's 8 groups of the box; the stage uses 4 of them
          const uint8_t *sb = smem + cslot * C::STAGE_BYTES + C::NMAT * BOX + row * 16 + (kb0 & 4) * 2;
#pragma unroll
          for (int mt = 0; mt < C::NMAT; ++mt) {
            sv[mt] = *reinterpret_cast<const uint2 *>(sb + mt * 2 * SBOX);
            bv[mt] = *reinterpret_cast<const uint2 *>(sb + mt * 2 * SBOX + SBOX);
          }
        }
        const uint8_t *stage = smem + cslot * C::STAGE_BYTES + row * 128;
        const int r7 = row & 7;
#pragma unroll 1
        for (int j = (int)((wg + NWG - kbc % NWG) % NWG); j < nkb; j += NWG) {
          const uint32_t kbg = kbc + j;
          const uint32_t aslot = kbg % NSLOT;
#pragma unroll
          for (int mat = 0; mat < C::NMAT; ++mat) {
            const uint8_t *rb = stage + mat * BOX;
            const uint4 w0 = *reinterpret_cast<const uint4 *>(rb + (((2 * j) ^ r7) << 4));
            const uint4 w1 = *reinterpret_cast<const uint4 *>(rb + (((2 * j + 1) ^ r7) << 4));
            const GroupScale gs = group_scale(pick_group(sv[mat], j), pick_group(bv[mat], j));
            uint32_t v[32];
            const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            if (gs.small) {  // the usual route (common.cuh)
#pragma unroll
              for (int wi = 0; wi < 8; ++wi) dq_word_small(wv[wi], gs, v + wi * 4);
            } else {
#pragma unroll
              for (int wi = 0; wi < 8; ++wi) dq_word_general(wv[wi], gs, v + wi * 4);
            }
            if (mat == 0) {  // the slot's previous k-block has left the MMA
              if (!__all_sync(0xffffffffu, timed(tr, w_free, [&] {
                    return wait_bar(&m->free[aslot], ((kbg / NSLOT) & 1u) ^ 1u, m, a.status);
                  }))) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
            }
            ptx::tmem_st_x32(tmem + lane_base + C::A_COL + aslot * C::A_SLOT + mat * 32, v);
          }
          if (!ok) break;
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&m->ready[aslot]);
        }
        kbc += nkb;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&m->code_empty[cslot]);
        if (!ok) break;
        // With one accumulator the previous item's epilogue runs once this
        // item's first stage is rebuilt: those k-blocks' ring slots were
        // freed by the previous item's MMAs (a stage fits the ring), so the
        // MMA finds them ready the moment the accumulator comes back.
        if (C::NBUF == 1 && st == 0 && has_prev) {
          if (!epilogue(prev, itc - 1)) break;
          has_prev = false;
        }
      }
      if (!ok) break;
      // With two accumulators the epilogue of an item runs after the next
      // item's k-blocks have been rebuilt (the MMA has long finished it by
      // then).
      if (C::NBUF == 2 && has_prev && !epilogue(prev, itc - 1)) break;
      prev = it;
      has_prev = true;
      ++itc;
    }
    if (ok && has_prev) epilogue(prev, itc - 1);
    if (lane == 0) ptx::bulk_wait_all();  // the epilogue's stores have landed
    if (tr) {
      trace_put(a, TW_DQ_CODE, w_code);
      trace_put(a, TW_DQ_FREE, w_free);
      trace_put(a, TW_DQ_ACC, w_acc);
      trace_put(a, TW_DQ_TOTAL, (unsigned long long)(clock64() - t_start));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Token rows of the gate/up GEMM in block-map row order, interleaved along K
// (see ilv_pos): row p < k*T is x[perm[p] / k] (the routed pairs in perm
// order), row k*T + t is x[t] (the shared expert).  One warp per row, 16-byte
// loads and stores; each 8-value run (v0 .. v7) is stored as v0 v4 v1 v5 v2
// v6 v3 v7.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t *__restrict__ x,
                                                          const int32_t *__restrict__ perm, int routed, int rows,
                                                          int k, int K, uint16_t *__restrict__ xg) {
  // launched as a programmatic dependent of the scatter: its perm first; the
  // gate/up kernel that follows may be scheduled from here on (it waits for
  // this grid's rows before it reads them)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int t = r < routed ? perm[r] / k : r - routed;
  const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * K);
  uint4 *dst = reinterpret_cast<uint4 *>(xg + (size_t)r * K);
  for (int i = lane; i < K / 8; i += 32) {
    const uint4 v = __ldg(src + i);
    dst[i] = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632), __byte_perm(v.y, v.w, 0x5410),
                        __byte_perm(v.y, v.w, 0x7632));
  }
}

// ---------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

// Scales or biases as a 2D bf16 tensor [rows_total][K/64], boxes of 128 rows x
// 8 groups (16 bytes), no swizzle.
cudaError_t group_map(CUtensorMap *map, const uint16_t *p, int rows_total, int K) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorInitializationError;
  cuuint64_t dims[2] = {(cuuint64_t)(K / KBLK), (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {(cuuint64_t)(K / KBLK) * 2};
  cuuint32_t box[2] = {8, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(p), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Packed codes as a 2D byte tensor [rows_total][K/2], boxes of 128 x 128 B.
cudaError_t code_map(CUtensorMap *map, const uint32_t *codes, int rows_total, int K) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorInitializationError;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t *>(codes), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Output rows (h or y) as a 2D bf16 tensor [rows_total][NOUT], boxes of 32
// features x 16 rows, no swizzle (the epilogue's staging layout).
cudaError_t out_map(CUtensorMap *map, const uint16_t *p, int rows_total, int NOUT) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorInitializationError;
  cuuint64_t dims[2] = {(cuuint64_t)NOUT, (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {(cuuint64_t)NOUT * 2};
  cuuint32_t box[2] = {32, 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Activation rows as a 2D bf16 tensor [rows_total][K], boxes of one k-block
// (64 values, 128 B) x box_rows rows, 128B swizzle (the MMA's K-major layout).
cudaError_t act_map(CUtensorMap *map, const uint16_t *p, int rows_total, int K, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorInitializationError;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows_total};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)KBLK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// One launch of the grouped kernel; with pdl, as a programmatic dependent of
// the kernel before it in the stream.
template <int MODE>
cudaError_t launch_tc(const TcMaps &m, const TcArgs &a, int grid, bool pdl, cudaStream_t s) {
  return launch_dep(pdl, experts_tc_kernel<MODE>, dim3(grid), dim3(THREADS), Cfg<MODE>::SMEM, s, m, a);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool tc_supported(const moe_config &c) { return c.hidden % 256 == 0 && c.inter % 256 == 0; }

cudaError_t tc_prepare() {
  cudaError_t e = cudaFuncSetAttribute(experts_tc_kernel<MODE_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<MODE_GATEUP>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(experts_tc_kernel<MODE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<MODE_DOWN>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(experts_tc_kernel<MODE_DOWN2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<MODE_DOWN2>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(experts_tc_kernel<MODE_DOWN2_SHORT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<MODE_DOWN2_SHORT>::SMEM);
  return e;
}

cudaError_t launch_experts_tc(const moe_plan_t *plan, const uint16_t *x, int T, const int32_t *perm,
                              const int32_t *blockmap, const int32_t *n_tiles, int max_tiles, int down_mode,
                              const int32_t *blockmap2, const int32_t *n_tiles2, int max_tiles2, ExpertPtrs w,
                              uint16_t *h, uint16_t *y, uint16_t *xg, int32_t *qctr, int32_t *status,
                              uint64_t *trace, int *launches, cudaStream_t s) {
  const moe_config &c = plan->cfg;
  const int rows_gu = (c.n_experts + c.n_shared) * c.inter;
  const int rows_dn = (c.n_experts + c.n_shared) * c.hidden;
  TcMaps mg{}, md{};
  cudaError_t e;
  // Each grouped kernel starts as a programmatic dependent of the kernel
  // before it (the gather, then gate/up) unless a timing event sits between.
  bool gather_quiet = true;
  const bool ts_gu = c.hidden % 512 == 0, ts_dn = c.inter % 512 == 0;
  if ((e = code_map(&mg.code[0], w.gate_q, rows_gu, c.hidden)) != cudaSuccess) return e;
  if ((e = code_map(&mg.code[1], w.up_q, rows_gu, c.hidden)) != cudaSuccess) return e;
  if ((e = code_map(&md.code[0], w.down_q, rows_dn, c.inter)) != cudaSuccess) return e;
  if (ts_gu) {
    if ((e = group_map(&mg.sc[0], w.gate_s, rows_gu, c.hidden)) != cudaSuccess) return e;
    if ((e = group_map(&mg.bi[0], w.gate_b, rows_gu, c.hidden)) != cudaSuccess) return e;
    if ((e = group_map(&mg.sc[1], w.up_s, rows_gu, c.hidden)) != cudaSuccess) return e;
    if ((e = group_map(&mg.bi[1], w.up_b, rows_gu, c.hidden)) != cudaSuccess) return e;
  }
  if (ts_dn) {
    if ((e = group_map(&md.sc[0], w.down_s, rows_dn, c.inter)) != cudaSuccess) return e;
    if ((e = group_map(&md.bi[0], w.down_b, rows_dn, c.inter)) != cudaSuccess) return e;
  }
  // two output tiles per down item: both "matrices" are the down weights
  md.code[1] = md.code[0];
  md.sc[1] = md.sc[0];
  md.bi[1] = md.bi[0];
  // h: the routed rows (k per token) then the shared expert's (n_shared per token)
  const int rows_h = (c.top_k + c.n_shared) * T;
  for (int i = 0; i < 4; ++i)
    if ((e = act_map(&md.act[i], h, rows_h, c.inter, BM >> i)) != cudaSuccess) return e;
  if ((e = out_map(&mg.out, h, rows_h, c.inter)) != cudaSuccess) return e;
  if ((e = out_map(&md.out, y, rows_h, c.hidden)) != cudaSuccess) return e;
  {  // gate/up token rows by TMA from a gathered, interleaved copy of x
    for (int i = 0; i < 4; ++i)
      if ((e = act_map(&mg.act[i], xg, rows_h, c.hidden, BM >> i)) != cudaSuccess) return e;
    gather_quiet = prof_quiet(MOE_KERNEL_GATHER);
    const bool pdl = prof_chain(MOE_KERNEL_GATHER);  // a dependent of the scatter
    prof_before(MOE_KERNEL_GATHER, s);
    e = launch_dep(pdl, gather_rows_kernel, dim3((rows_h + 7) / 8), dim3(256), 0, s, x, perm, c.top_k * T, rows_h,
                   c.top_k, c.hidden, xg);
    prof_after(MOE_KERNEL_GATHER, s);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    *launches += 1;
  }

  TcArgs a{};
  a.blockmap = blockmap;
  a.n_tiles = n_tiles;
  a.item_counter = qctr;  // gate/up's queue (the scatter kernel zeroed both)
  a.status = status;
  a.T = T;
  a.k = c.top_k;
  a.E = c.n_experts;
  a.trace = trace;
  a.trace_base = 0;

  // gate/up + SwiGLU: x rows (gathered) -> h
  a.sc[0] = w.gate_s;
  a.bi[0] = w.gate_b;
  a.sc[1] = w.up_s;
  a.bi[1] = w.up_b;
  a.out = h;
  a.K = c.hidden;
  a.NOUT = c.inter;
  a.tma_scales = ts_gu;
  a.first = c.n_shared ? (T + plan->block_rows - 1) / plan->block_rows : 0;
  int items = max_tiles * (c.inter / BM);
  int grid = items < plan->num_sms ? items : plan->num_sms;
  const bool gu_quiet = prof_quiet(MOE_KERNEL_GATEUP);
  prof_before(MOE_KERNEL_GATEUP, s);
  e = launch_tc<MODE_GATEUP>(mg, a, grid, gather_quiet && gu_quiet, s);
  prof_after(MOE_KERNEL_GATEUP, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // down: h rows -> y, in the mode the caller chose (tc.h)
  const bool first_map = down_mode == TC_DOWN_PAIR;
  const bool pair = down_mode != TC_DOWN_ONE;
  a.trace_base = 16;
  a.blockmap = first_map ? blockmap : blockmap2;
  a.n_tiles = first_map ? n_tiles : n_tiles2;
  a.item_counter = qctr + 1;  // down's queue (the scatter kernel zeroed it)
  a.sc[0] = w.down_s;
  a.bi[0] = w.down_b;
  a.sc[1] = w.down_s;
  a.bi[1] = w.down_b;
  a.out = y;
  a.K = c.inter;
  a.NOUT = c.hidden;
  a.tma_scales = ts_dn;
  {
    const int bn = first_map ? plan->block_rows : down_mode == TC_DOWN_PAIR_SHORT ? TC_SHORT_ROWS : plan->block_rows2;
    a.first = c.n_shared ? (T + bn - 1) / bn : 0;
  }
  items = (first_map ? max_tiles : max_tiles2) * (c.hidden / ((pair ? 2 : 1) * BM));
  grid = items < plan->num_sms ? items : plan->num_sms;
  const bool dn_pdl = gu_quiet && prof_quiet(MOE_KERNEL_DOWN);
  prof_before(MOE_KERNEL_DOWN, s);
  e = down_mode == TC_DOWN_PAIR         ? launch_tc<MODE_DOWN2>(md, a, grid, dn_pdl, s)
      : down_mode == TC_DOWN_PAIR_SHORT ? launch_tc<MODE_DOWN2_SHORT>(md, a, grid, dn_pdl, s)
                                        : launch_tc<MODE_DOWN>(md, a, grid, dn_pdl, s);
  prof_after(MOE_KERNEL_DOWN, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  *launches += 2;
  return cudaSuccess;
}

}  // namespace moe
