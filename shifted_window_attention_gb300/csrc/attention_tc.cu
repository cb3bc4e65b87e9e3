// Tensor-core window attention for sm_103a: bf16 Q/K/V, fp32 accumulation and
// softmax, bf16 output.
//
// What it computes ("Window-Aligned Sequence Parallelism (SeedVR2)", section
// "Motivation"): for every window w of a plan and every head h,
//     O[w,h] = softmax(Q[w,h] K[w,h]^T * scale) V[w,h],
// attention only inside the window.  Rows of a window are gathered from the
// token-major [N, heads, 128] tensors through the plan's ids table and the
// output rows are scattered back through it, so no separate permutation pass
// touches HBM.
//
// Design (Blackwell, one CTA per SM, persistent):
//  * A work unit is (window, head, 256 query rows) -- two 128-row Q tiles that
//    share every K/V tile, halving K/V traffic per FLOP.  Units are handed out
//    by an atomic counter in heaviest-first order (the note's LPT rule applied
//    to kernel work units), so ragged edge windows fill the tail.
//  * Warp roles: warps 0-3 run the softmax of Q tile 0 and warps 4-7 that of
//    Q tile 1 (one query row per thread = one TMEM lane); warps 8-9 gather
//    Q/K/V rows with 16-byte cp.async into 128B-swizzled shared-memory tiles;
//    warp 10 issues every tcgen05.mma (the warp converged, one elected lane
//    issuing each group of 8 with its commits), and one thread of warp 11
//    takes work units from the global counter up to two units ahead.
//  * Rows in plan-packed order: a full 128-row tile of a window is a plain
//    strided block of the [N, heads, 128] tensor, so it arrives by two TMA
//    tile loads (cp.async.bulk.tensor, one per 64-channel panel, the same
//    128-byte swizzle).  A window's last, partial tile is still gathered with
//    zero fill, so no row of another window ever enters a tile.
//  * TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  The bf16
//    probabilities P overwrite the first 64 columns of their S tile and feed
//    the P V product straight from TMEM (A operand in TMEM); V is the B
//    operand, read MN-major from shared memory.
//  * Online softmax in the log2 domain with a lazy rescale: the running max is
//    only raised (and O rescaled in TMEM) when a row's max grows by more than
//    64 (log2), which keeps every probability <= 2^64 and the result exact up
//    to rounding.  The row sum accumulates the same bf16-rounded probabilities
//    that enter the P V product.
//  * Output rows leave TMEM through registers with 256-bit stores when the
//    output is 32-byte aligned.
//  * Every wait is bounded: after ~1 s a wait records an error code in the
//    plan's workspace and the CTA unwinds, drains its MMAs and cp.asyncs and
//    frees TMEM.

#include <cuda.h>  // CUtensorMap and its encoder's types (the encoder is reached through the runtime)
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "wsa_internal.h"

namespace wsa {
namespace {

constexpr int kD = 128;                     // head dim
constexpr int kTile = 128;                  // rows of a Q / K / V tile
constexpr int kTileBytes = kTile * kD * 2;  // 32 KB
constexpr int kPanelBytes = kTile * 128;    // 128 rows x 128 B (64 channels), one swizzle panel
constexpr int kSlots = 5;                   // K/V ring slots
constexpr int kLoaderWarp0 = 8;
constexpr int kLoaderWarps = 2;
constexpr int kLoaderRows = kTile / kLoaderWarps;  // 64 rows of each tile per gather warp
constexpr int kIdsPerLane = kLoaderRows / 32;      // row ids a lane holds for one tile
constexpr int kMmaWarp = kLoaderWarp0 + kLoaderWarps;
constexpr int kSchedWarp = kMmaWarp + 1;
constexpr int kThreads = (kSchedWarp + 1) * 32;     // 12 warps: 3 per SM sub-partition
// Lazy-rescale threshold (log2).  Probabilities stay <= 2^64 (bf16 reaches
// 2^127); a row sum over at most 2^12 keys stays <= 2^76 and O <= 2^76 max|v|,
// far inside fp32, and O and the sum carry the same scale, so the relative
// precision does not depend on it.  Measured: 1080p (outlier channels, frequent
// max jumps) 1077 / 1064 TFLOP/s at 24 and 1167 / 1152 at 64, 720p and the
// long clip unchanged; 8 cost 1080p a further 17%.
constexpr float kRescaleLog2 = 64.0f;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr long long kTmaDrainCycles = 400000LL;  // ~0.2 ms: TMA loads in flight after an error

enum : int {
  B_RING_FULL = 0,
  B_RING_EMPTY = B_RING_FULL + kSlots,
  B_Q_FULL = B_RING_EMPTY + kSlots,
  B_Q_EMPTY,
  B_S_FULL,                    // 2
  B_P_FULL = B_S_FULL + 2,     // 2
  B_O_FULL = B_P_FULL + 2,     // 2
  B_UNIT_FULL = B_O_FULL + 2,  // 2
  B_UNIT_EMPTY = B_UNIT_FULL + 2,
  B_DRAIN = B_UNIT_EMPTY + 2,
  B_COUNT
};

constexpr int kSmemQ = 0;                                   // Q0 | Q1
constexpr int kSmemRing = 2 * kTileBytes;                   // kSlots K/V tiles
constexpr int kSmemBars = kSmemRing + kSlots * kTileBytes;  // mbarriers
constexpr int kSmemUnits = kSmemBars + ((8 * B_COUNT + 15) / 16) * 16;
constexpr int kSmemTmem = kSmemUnits + 2 * 16;
constexpr int kSmemUsed = kSmemTmem + 16;
constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack for 1 KB alignment of the tiles

constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
constexpr uint32_t kTmemCols = 512;

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), A K-major (bit 15 = 0), N>>3 at bits 17-22, M>>4 at 24-28.
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
// P V: B (= V) is MN-major (bit 16).
constexpr uint32_t kIdescPV = kIdescS | (1u << 16);

// Error codes recorded in the workspace error word (which wait gave up).
enum : int {
  E_LOAD_UNIT_EMPTY = 0x101, E_LOAD_UNIT_FULL, E_LOAD_Q_EMPTY, E_LOAD_RING_EMPTY, E_SCHED_UNIT_EMPTY,
  E_MMA_UNIT_FULL = 0x201, E_MMA_Q_FULL, E_MMA_K_FULL, E_MMA_V_FULL, E_MMA_P0, E_MMA_P1, E_MMA_DRAIN,
  E_SM_UNIT_FULL = 0x301, E_SM_S_FULL, E_SM_O_FULL
};

struct TcParams {
  // Tile maps of q, k, v as [N rows][heads][128] bf16, box 64 channels x 1
  // head x 128 rows, 128-byte swizzle (set only for the packed-order TMA path).
  CUtensorMap tm_q, tm_k, tm_v;
  const char* q;
  const char* k;
  const char* v;
  char* o;
  const int* row_map;  // ids table (canonical order) or nullptr (packed order)
  const int* offsets;
  const WorkItem* items;
  int num_units;
  int heads;
  int n_tokens;          // rows of q, k, v, o (bound of every ids entry)
  // Text segment (n_text = 0: video only).  Window w's attention runs over the
  // segment [its n_w video rows, the n_text text rows]; text query rows write
  // fp32 partials T_w / W to text_part[w][t][head][128].  The segment is tiled
  // as the video rows' ceil(n_w/128) tiles followed by the text rows'
  // ceil(n_text/128) tiles, so that every tile has a single row source.
  const char* qt;
  const char* kt;
  const char* vt;
  float* text_part;
  int n_text;
  float inv_windows;
  long long row_stride;  // bytes between consecutive tokens (heads * 256)
  float c;               // softmax scale * log2(e)
  int o_v8;              // output rows 32-byte aligned: 256-bit stores
  int withhold_units;    // failure-path test hook: hand out no work unit
  int* work;             // workspace words
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Gives up when another thread has
// recorded an error, or after kWaitCycles, recording `code` first.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int* err, int code) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*reinterpret_cast<volatile int*>(err) != 0) return false;
      if (clock64() - t0 > kWaitCycles) {
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}

// Raises the transaction count the barrier's current phase waits for (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// TMA tile load of box (x, y, z) of a 3-D tensor map into shared memory; the
// landed bytes complete transactions on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrives on `bar` once every cp.async issued so far by this thread has
// landed (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Makes this thread's completed generic-proxy shared-memory writes visible to
// the async proxy (the tensor core reads its operands through it).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrives on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// One lane of a converged warp (elect.sync: the same lane every time for a
// full mask, so its commits track its own MMAs).
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile("{\n\t.reg .pred P;\n\t.reg .b32 R;\n\telect.sync R|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}"
               : "=r"(p));
  return p != 0;
}

// Shared-memory matrix descriptor: start address, leading/stride byte offsets
// (16-byte units), version 1 (bits 46-47), 128-byte swizzle (bits 61-63 = 2).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// K-major operand (Q or K tile, 128 rows x 128 channels): K-step kk covers
// channels 16kk..16kk+15: panel kk/4, 32-byte offset (kk%4) inside the
// swizzled 128-byte row; 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
  return smem_desc(tile + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
}

// MN-major B operand (V tile: K = key rows, N = channels): K-step kk covers
// key rows 16kk..16kk+15 (two 8-row groups 1024 bytes apart); the two
// 64-channel panels are kPanelBytes apart.
__device__ __forceinline__ uint64_t desc_v(uint32_t tile, int kk) {
  return smem_desc(tile + kk * 2048, kPanelBytes, 1024);
}

// The start-address field (bits 0-13, in 16-byte units) of the K-step kk
// descriptors above, relative to step 0: a descriptor of step kk is the step-0
// descriptor plus this constant (shared-memory addresses stay below 2^18, so
// the field never carries into the next one).
constexpr uint64_t kmajor_step(int kk) { return static_cast<uint64_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4); }
constexpr uint64_t v_step(int kk) { return static_cast<uint64_t>((kk * 2048) >> 4); }

#define WSA_R8(b) "=r"(r[b]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), "=r"(r[b + 5]), \
                  "=r"(r[b + 6]), "=r"(r[b + 7])
#define WSA_W8(b) "r"(r[b]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), "r"(r[b + 4]), "r"(r[b + 5]), \
                  "r"(r[b + 6]), "r"(r[b + 7])

// 64 consecutive fp32 columns of this thread's TMEM lane; the wait is inside
// the same asm statement so no use of the registers can be scheduled before it.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,"
      "%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,"
      "%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : WSA_R8(0), WSA_R8(8), WSA_R8(16), WSA_R8(24), WSA_R8(32), WSA_R8(40), WSA_R8(48), WSA_R8(56)
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(r[i]);
}

// 128 consecutive fp32 columns in one load (one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&x)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : WSA_R8(0), WSA_R8(8), WSA_R8(16), WSA_R8(24), WSA_R8(32), WSA_R8(40), WSA_R8(48), WSA_R8(56),
        WSA_R8(64), WSA_R8(72), WSA_R8(80), WSA_R8(88), WSA_R8(96), WSA_R8(104), WSA_R8(112), WSA_R8(120)
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&x)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,"
      "%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : WSA_R8(0), WSA_R8(8), WSA_R8(16), WSA_R8(24)
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,"
      "%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      WSA_W8(0), WSA_W8(8), WSA_W8(16), WSA_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      WSA_W8(0), WSA_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------- roles

struct Smem {
  uint32_t q0, ring, bars;
  int4* units;
};

__device__ __forceinline__ uint32_t bar_at(const Smem& s, int i) { return s.bars + 8u * static_cast<uint32_t>(i); }

// Gather warps (2): rows 64*lw .. 64*lw+63 of every tile.  A half-warp copies
// one 256-byte row (16 chunks of 16 bytes), so each lane issues 32 cp.async
// per tile, each addressed by one 32 x 32 -> 64-bit multiply-add.  These warps
// share their sub-partitions with four of the softmax warps, whose issue slots
// they take: the short address path measured 5-6% faster than a 64-bit
// multiply and two selects per copy.  Shared layout: two 64-channel panels of 128 rows x 128 bytes,
// chunk c of row r stored at chunk position c ^ (r % 8) (128-byte swizzle).
// Completion is signalled asynchronously: after its copies for a tile, every
// lane arms a cp.async arrive on the tile's full barrier (64 arrivals), so the
// gather warps never wait for data; the MMA warp makes the landed rows
// visible to the tensor core with a proxy fence.  The token ids of the next
// key tile are fetched while the current one is issued.
// kTma (packed rows, no text): full tiles come by TMA instead.  Lane 0 of
// gather warp 0 raises the barrier's transaction count by the tile's bytes
// and issues the two panel loads; every lane still makes its usual arrival,
// so the barrier counts are the same for both kinds of tile.
template <bool kText, bool kTma>
__device__ __forceinline__ void loader_role(const TcParams& prm, const Smem& sm, int lw, int lane) {
  int* err = prm.work + WS_ERROR;
  const int half = lane >> 4;
  const int chunk = lane & 15;
  const uint32_t panel_off = static_cast<uint32_t>((chunk >> 3) * kPanelBytes);
  const int cc = chunk & 7;
  uint32_t ring_iter = 0, unit_iter = 0;

  auto acquire = [&](uint32_t bar, uint32_t parity, int code) -> bool {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, err, code));
  };
  // lane l holds the source rows of rows kLoaderRows*lw + 32*h + l of segment
  // tile j (-1: past the end of its part, zero fill): a video row id for the
  // first nvt tiles, a text row index for the text tiles after them.
  auto fetch_ids = [&](int (&ids)[kIdsPerLane], int j, int nv, int nvt, int off) {
#pragma unroll
    for (int h = 0; h < kIdsPerLane; ++h) {
      const int lr = kLoaderRows * lw + 32 * h + lane;
      ids[h] = -1;
      if (!kText || j < nvt) {
        const int myrow = j * kTile + lr;
        if (myrow < nv) {
          int id = prm.row_map ? __ldg(prm.row_map + off + myrow) : off + myrow;
          if (kBoundsCheck && static_cast<unsigned>(id) >= static_cast<unsigned>(prm.n_tokens)) {
            atomicCAS(prm.work + WS_BOUNDS, 0, kErrBounds);
            id = -1;  // read as zeros
          }
          ids[h] = id;
        }
      } else {
        const int tr = (j - nvt) * kTile + lr;
        if (tr < prm.n_text) ids[h] = tr;
      }
    }
  };
  auto copy_tile = [&](const char* src, uint32_t dst, const int (&ids)[kIdsPerLane], int head) {
    const uint64_t colbase = reinterpret_cast<uint64_t>(src) + static_cast<uint64_t>(head) * (kD * 2) + chunk * 16;
    const uint32_t stride = static_cast<uint32_t>(prm.row_stride);  // heads * 256 < 2^24
#pragma unroll
    for (int i = 0; i < kLoaderRows / 2; ++i) {
      const int r = kLoaderRows * lw + half + 2 * i;
      const int id = __shfl_sync(0xffffffffu, ids[i >> 4], half + 2 * (i & 15));
      // a row past the end (id -1) reads row 0 with source size 0 (zero fill):
      // one 32 x 32 -> 64-bit multiply-add per copy
      const uint32_t row = static_cast<uint32_t>(max(id, 0));
      const uint64_t g = colbase + static_cast<uint64_t>(row) * stride;
      cp_async16(dst + panel_off + r * 128 + ((cc ^ (r & 7)) << 4), reinterpret_cast<const void*>(g),
                 id >= 0 ? 16u : 0u);
    }
  };
  const bool tma_lane = kTma && lw == 0 && lane == 0;
  // Which of the latest ring fills came by TMA (bit i: fill ring_iter - 1 -
  // i), and the latest Q fill when it did (unit iteration + 1, else 0).  A
  // slot is refilled only after its previous fill was consumed, so after an
  // error only the last kSlots fills and the last Q fill can still be landing.
  uint32_t tma_bits = 0, tma_q = 0;
  // Both panels of the packed rows [row, row + 128) of `head` (TMA path only).
  auto tma_tile = [&](const CUtensorMap* map, uint32_t dst, int row, int head, uint32_t bar) {
    mbar_expect_tx(bar, kTileBytes);
    tma_load_3d(dst, map, 0, head, row, bar);
    tma_load_3d(dst + kPanelBytes, map, 64, head, row, bar);
  };
  // text: a text tile; tma_row >= 0: a full tile of packed rows from that row
  auto load_kv = [&](const int (&ids)[kIdsPerLane], int head, bool text, int tma_row) -> bool {
    for (int which = 0; which < 2; ++which) {
      const uint32_t slot = ring_iter % kSlots;
      if (!acquire(bar_at(sm, B_RING_EMPTY + slot), ((ring_iter / kSlots) & 1) ^ 1, E_LOAD_RING_EMPTY))
        return false;
      const uint32_t full = bar_at(sm, B_RING_FULL + slot);
      if (kTma) tma_bits = (tma_bits << 1) | (tma_row >= 0 ? 1u : 0u);
      if (kTma && tma_row >= 0) {
        if (tma_lane) tma_tile(which ? &prm.tm_v : &prm.tm_k, sm.ring + slot * kTileBytes, tma_row, head, full);
      } else {
        copy_tile(kText && text ? (which ? prm.vt : prm.kt) : (which ? prm.v : prm.k), sm.ring + slot * kTileBytes,
                  ids, head);
      }
      cp_async_arrive(full);
      ++ring_iter;
    }
    return true;
  };
  // Packed row of tile j when it is a full tile loaded by TMA, else -1.
  auto tma_row_of = [&](int j, int nv, int off) -> int {
    return kTma && (j + 1) * kTile <= nv ? off + j * kTile : -1;
  };

  while (true) {
    const int us = unit_iter & 1;
    const uint32_t uph = (unit_iter >> 1) & 1;
    if (!acquire(bar_at(sm, B_UNIT_FULL + us), uph, E_LOAD_UNIT_FULL)) break;
    const int4 info = sm.units[us];
    if (info.y < 0) break;
    const int off = info.x, nv = info.y, q0 = info.z, head = info.w & 0xffff;
    const int nvt = (nv + kTile - 1) / kTile;
    const int nkv = nvt + (kText ? (prm.n_text + kTile - 1) / kTile : 0);
    const int qt0 = q0 / kTile;
    const bool has1 = qt0 + 1 < nkv;
    int ids[kIdsPerLane], ids_next[kIdsPerLane], qids0[kIdsPerLane], qids1[kIdsPerLane];
    fetch_ids(ids, 0, nv, nvt, off);
    fetch_ids(qids0, qt0, nv, nvt, off);
    if (has1) fetch_ids(qids1, qt0 + 1, nv, nvt, off);
    // K0/V0 first: they may land while the previous unit's last MMAs still
    // hold the Q buffers.
    if (nkv > 1) fetch_ids(ids_next, 1, nv, nvt, off);
    if (!load_kv(ids, head, nvt == 0, tma_row_of(0, nv, off))) break;
    if (!acquire(bar_at(sm, B_Q_EMPTY), (unit_iter & 1) ^ 1, E_LOAD_Q_EMPTY)) break;
    const uint32_t qfull = bar_at(sm, B_Q_FULL);
    const int qrow0 = tma_row_of(qt0, nv, off), qrow1 = has1 ? tma_row_of(qt0 + 1, nv, off) : -1;
    if (kTma) tma_q = qrow0 >= 0 || qrow1 >= 0 ? unit_iter + 1 : 0;
    if (kTma && qrow0 >= 0) {
      if (tma_lane) tma_tile(&prm.tm_q, sm.q0, qrow0, head, qfull);
    } else {
      copy_tile(kText && qt0 >= nvt ? prm.qt : prm.q, sm.q0, qids0, head);
    }
    if (kTma && qrow1 >= 0) {
      if (tma_lane) tma_tile(&prm.tm_q, sm.q0 + kTileBytes, qrow1, head, qfull);
    } else if (has1) {
      copy_tile(kText && qt0 + 1 >= nvt ? prm.qt : prm.q, sm.q0 + kTileBytes, qids1, head);
    }
    cp_async_arrive(qfull);
    bool ok = true;
    for (int j = 1; j < nkv && ok; ++j) {
#pragma unroll
      for (int h = 0; h < kIdsPerLane; ++h) ids[h] = ids_next[h];
      if (j + 1 < nkv) fetch_ids(ids_next, j + 1, nv, nvt, off);
      ok = load_kv(ids, head, j >= nvt, tma_row_of(j, nv, off));
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_at(sm, B_UNIT_EMPTY + us));
    ++unit_iter;
  }
  cp_async_wait_all();
  // After a failed wait, TMA loads this lane issued may still be landing.
  // Wait for the barrier phase of each fill that came by TMA (every lane
  // arrived on it right after the load was issued, so it completes when the
  // bytes have landed), bounded and regardless of the error word.  A phase
  // that does not complete in time (another gather warp gave up before its
  // arrival) leaves a fixed bounded wait as the last resort before the CTA
  // releases its shared memory.
  if (tma_lane && *reinterpret_cast<volatile int*>(err) != 0) {
    const long long t0 = clock64();
    auto drained = [&](uint32_t bar, uint32_t parity) {
      while (!mbar_try(bar, parity))
        if (clock64() - t0 > kTmaDrainCycles) return false;
      return true;
    };
    bool ok = true;
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      if (i >= static_cast<int>(ring_iter) || !((tma_bits >> i) & 1u)) continue;
      const uint32_t f = ring_iter - 1 - i;
      ok = drained(bar_at(sm, B_RING_FULL + f % kSlots), (f / kSlots) & 1) && ok;
    }
    if (tma_q != 0) ok = drained(bar_at(sm, B_Q_FULL), (tma_q - 1) & 1) && ok;
    if (!ok)
      while (clock64() - t0 < 2 * kTmaDrainCycles) __nanosleep(1000);
  }
}

// One thread hands out work units: it takes the next unit from the global
// counter as soon as a unit slot is free, so the next unit's description is
// ready (up to two units ahead) before the gather warps finish the current one.
__device__ __forceinline__ void scheduler_role(const TcParams& prm, const Smem& sm) {
  int* err = prm.work + WS_ERROR;
  // Test hook: with no unit published, every other role's first wait runs
  // out and the kernel unwinds with nothing in flight.
  if (prm.withhold_units) return;
  for (uint32_t unit_iter = 0;; ++unit_iter) {
    const int us = unit_iter & 1;
    if (!wait_bar(bar_at(sm, B_UNIT_EMPTY + us), ((unit_iter >> 1) & 1) ^ 1, err, E_SCHED_UNIT_EMPTY)) break;
    const int u = atomicAdd(prm.work + WS_NEXT_UNIT, 1);
    int4 info = make_int4(0, -1, 0, 0);
    if (u < prm.num_units) {
      const WorkItem it = prm.items[u / prm.heads];
      const int off = prm.offsets[it.window];
      info = make_int4(off, prm.offsets[it.window + 1] - off, it.q_start, (u % prm.heads) | (it.window << 16));
    }
    sm.units[us] = info;
    mbar_arrive(bar_at(sm, B_UNIT_FULL + us));
    if (info.y < 0) break;
  }
}

// The MMA warp issues every MMA.  Per key tile j:
//   S0 = Q0 K_j^T ; [PV1 of tile j-1] ; S1 = Q1 K_j^T ; PV0 of tile j
// so the softmax of one Q tile overlaps the MMAs of the other.  S_t of tile
// j+1 overwrites P_t of tile j only after PV_t(j) was issued (tcgen05.mma
// from one thread execute in order).  O0 is released to its epilogue right
// after the unit's last PV0, so that epilogue overlaps tile 1's last softmax
// and P V (bit-identical; 0.1-1.2% faster across the workloads).
// The whole warp runs the role converged: every lane waits and keeps the
// counters, and one elected lane (the same one each time, so its commits
// track its own MMAs) issues each group of 8 MMAs together with its fences
// and commits.  A lone issuing lane, with the other 31 lanes parked, issued
// each M128 N128 K16 product in 84-97 cycles against 64: its instructions
// wait for issue slots behind the two softmax warps of the sub-partition.
// Measured: 1176 / 1090 TFLOP/s canonical and 1342 / 1235 packed at 720p
// against 1165 / 1073 and 1317 / 1213 with the lone lane.
// Every descriptor is a step-0 descriptor plus a constant, computed once per
// kernel (Q) or per tile (K, V), which keeps the issue path between MMAs
// short (with the converged warp: 1196 / 1108 against 1169 / 1084 TFLOP/s
// canonical at 720p, 1188 / 1171 against 1164 / 1140 at 1080p).
template <bool kText>
__device__ __forceinline__ void mma_role(const TcParams& prm, const Smem& sm, uint32_t tmem) {
  int* err = prm.work + WS_ERROR;
  // every lane waits; the result is the same in all lanes
  auto wait_warp = [&](uint32_t bar, uint32_t parity, int code) -> bool {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, err, code));
  };
  const uint32_t tS0 = tmem + kColS0, tS1 = tmem + kColS1, tO0 = tmem + kColO0, tO1 = tmem + kColO1;
  const uint32_t sQ1 = sm.q0 + kTileBytes;
  const uint64_t dQ0 = desc_kmajor(sm.q0, 0), dQ1 = desc_kmajor(sQ1, 0);
  uint32_t ring_iter = 0, unit_iter = 0, p_cnt0 = 0, p_cnt1 = 0;
  // S_t = Q_t K^T over the 8 K-steps of the key tile at kt
  auto issue_s = [&](uint32_t tS, uint64_t dq, uint64_t dk) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mma_ss(tS, dq + kmajor_step(kk), dk + kmajor_step(kk), kIdescS, kk > 0);
  };
  // O_t (+)= P_t V over the 8 K-steps of the value tile at vt
  auto issue_pv = [&](uint32_t tO, uint32_t tP, uint64_t dv, bool acc_first) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mma_ts(tO, tP + 8 * kk, dv + v_step(kk), kIdescPV, (acc_first || kk > 0) ? 1u : 0u);
  };
  while (true) {
    const int us = unit_iter & 1;
    if (!wait_warp(bar_at(sm, B_UNIT_FULL + us), (unit_iter >> 1) & 1, E_MMA_UNIT_FULL)) break;
    const int4 info = sm.units[us];
    if (info.y < 0) break;
    const int q0 = info.z;
    const int nkv = (info.y + kTile - 1) / kTile + (kText ? (prm.n_text + kTile - 1) / kTile : 0);
    const bool has1 = q0 / kTile + 1 < nkv;
    bool ok = true;
    uint32_t vslot_prev = 0;
    uint64_t dV_prev = 0;
    for (int j = 0; j < nkv; ++j) {
      const uint32_t kslot = ring_iter % kSlots;
      if (!(ok = wait_warp(bar_at(sm, B_RING_FULL + kslot), (ring_iter / kSlots) & 1, E_MMA_K_FULL))) break;
      if (j == 0 && !(ok = wait_warp(bar_at(sm, B_Q_FULL), unit_iter & 1, E_MMA_Q_FULL))) break;
      const uint32_t kt = sm.ring + kslot * kTileBytes;
      const uint64_t dK = desc_kmajor(kt, 0);
      if (elect_one()) {
        fence_proxy_async();  // rows landed by cp.async -> visible to the tensor core
        tc_fence_after();
        issue_s(tS0, dQ0, dK);
        tc_commit(bar_at(sm, B_S_FULL + 0));
      }
      __syncwarp();
      if (j > 0 && has1) {
        if (!(ok = wait_warp(bar_at(sm, B_P_FULL + 1), p_cnt1 & 1, E_MMA_P1))) break;
        ++p_cnt1;
      }
      if (elect_one()) {
        if (j > 0) {
          if (has1) {
            tc_fence_after();
            issue_pv(tO1, tS1, dV_prev, j > 1);
          }
          tc_commit(bar_at(sm, B_RING_EMPTY + vslot_prev));
        }
        if (has1) {
          issue_s(tS1, dQ1, dK);
          tc_commit(bar_at(sm, B_S_FULL + 1));
        }
        tc_commit(bar_at(sm, B_RING_EMPTY + kslot));
        if (j == nkv - 1) tc_commit(bar_at(sm, B_Q_EMPTY));
      }
      __syncwarp();
      ++ring_iter;
      const uint32_t vslot = ring_iter % kSlots;
      if (!(ok = wait_warp(bar_at(sm, B_RING_FULL + vslot), (ring_iter / kSlots) & 1, E_MMA_V_FULL))) break;
      if (!(ok = wait_warp(bar_at(sm, B_P_FULL + 0), p_cnt0 & 1, E_MMA_P0))) break;
      ++p_cnt0;
      const uint32_t vt = sm.ring + vslot * kTileBytes;
      const uint64_t dV = desc_v(vt, 0);
      if (elect_one()) {
        fence_proxy_async();
        tc_fence_after();
        issue_pv(tO0, tS0, dV, j > 0);
        if (j == nkv - 1) tc_commit(bar_at(sm, B_O_FULL + 0));
      }
      __syncwarp();
      ++ring_iter;
      dV_prev = dV;
      vslot_prev = vslot;
    }
    if (!ok) break;
    if (has1) {
      if (!wait_warp(bar_at(sm, B_P_FULL + 1), p_cnt1 & 1, E_MMA_P1)) break;
      ++p_cnt1;
    }
    if (elect_one()) {
      if (has1) {
        tc_fence_after();
        issue_pv(tO1, tS1, dV_prev, nkv > 1);
      }
      tc_commit(bar_at(sm, B_RING_EMPTY + vslot_prev));
      if (has1) tc_commit(bar_at(sm, B_O_FULL + 1));
      mbar_arrive(bar_at(sm, B_UNIT_EMPTY + us));
    }
    __syncwarp();
    ++unit_iter;
  }
  // Drain: every MMA issued so far must finish before TMEM is freed, also
  // when another role has given up (MMAs depend on nothing but their
  // operands, so this wait ends unless the tensor core itself has stopped).
  if (elect_one()) tc_commit(bar_at(sm, B_DRAIN));
  __syncwarp();
  const long long t0 = clock64();
  while (!mbar_try(bar_at(sm, B_DRAIN), 0)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicCAS(err, 0, E_MMA_DRAIN);
      break;
    }
  }
  __syncwarp();
}

// 32 bytes in one store (the address must be 32-byte aligned).  Output rows
// are not read again by this kernel, so they do not allocate in L1 (measured
// 1-2% faster than the default policy on every workload).
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                             uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
               "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// 16 bytes, same policy (outputs that are not 32-byte aligned).
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
  asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2), "r"(a3)
               : "memory");
}

// acc.x += lo(w), acc.y += hi(w) for the two bf16 halves of w, in fp32
// (the conversion of a bf16 to fp32 is exact, so the sums are those of the
// unpacked values).
__device__ __forceinline__ void add_bf16x2_f32(float2& acc, uint32_t w) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One key tile of the online softmax for this thread's query row: reads the
// 128 scores of S, updates the running max m (log2 domain, lazily) and the
// running sum l2 (two partial sums), rescales O in TMEM when the max grows by
// more than kRescaleLog2 (log2), and writes the bf16 probabilities P over the first 64
// columns of S.  kFull: all 128 key columns are valid (no masking).
// A full key tile whose row max grew past the threshold in some row of the
// warp: the max-first order (max, rescale of O and the sums, exponentials),
// reading S in 32-column pieces.  Piece h's P lands in columns 16h..16h+15,
// whose scores were read by then; the sums take the pairs in the same order.
__device__ __forceinline__ void softmax_tile_redo(uint32_t tS, uint32_t tO, float c, float& m, float2& la,
                                                  float2& lb) {
  float mx = -INFINITY;
#pragma unroll 1
  for (int h = 0; h < 4; ++h) {
    float y[32];
    tmem_ld32(tS + 32 * h, y);
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, y[i]);
  }
  const float m_new = fmaxf(m, mx * c);
  const float alpha = ex2(m - m_new);
  la = __fmul2_rn(la, make_float2(alpha, alpha));
  lb = __fmul2_rn(lb, make_float2(alpha, alpha));
  m = m_new;
#pragma unroll 1
  for (int h = 0; h < 4; ++h) {
    float o[32];
    tmem_ld32(tO + 32 * h, o);
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(o[i] * alpha);
    tmem_st32(tO + 32 * h, r);
  }
  tmem_wait_st();
  const float2 cc = make_float2(c, c);
  const float2 nm = make_float2(-m, -m);
#pragma unroll 1
  for (int h = 0; h < 4; ++h) {
    float y[32];
    tmem_ld32(tS + 32 * h, y);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 a = __ffma2_rn(make_float2(y[2 * i], y[2 * i + 1]), cc, nm);
      pk[i] = pack_bf16(ex2(a.x), ex2(a.y));
      if (i & 1) add_bf16x2_f32(lb, pk[i]); else add_bf16x2_f32(la, pk[i]);
    }
    tmem_st16(tS + 16 * h, pk);
  }
}

// kSpec (the TMA instantiation): full tiles after the first take the
// exponentials of their first half at the current running max while the row
// max is found alongside (below); the gather instantiation, where it measured
// slower, finds the max first.
template <bool kFull, bool kSpec>
__device__ __forceinline__ void softmax_tile(uint32_t tS, uint32_t tO, bool first, int kv_valid, float c,
                                             float& m, float2& la, float2& lb) {
  float x[128];
  tmem_ld128(tS, x);
  if (kSpec && kFull && !first) {
    // The running max moves only when a row max exceeds it by more than
    // kRescaleLog2, so the first half's exponentials are taken with the
    // current max while the row max is found alongside them, off the path
    // from S to P.  When the check calls for a rescale (rare), nothing has
    // been stored or summed yet, and the tile is redone from S (still intact
    // in TMEM) in 32-column pieces, in the same order as the max-first path:
    // the same bits, and few registers, so the common path keeps all of its.
    const float2 cc = make_float2(c, c);
    const float2 nm = make_float2(-m, -m);
    uint32_t pk[32];
    float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[64], x[65]);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = 2 * i;
      if (i > 0) {
        m0 = fmax3(m0, x[e], x[e + 1]);
        m1 = fmax3(m1, x[64 + e], x[65 + e]);
      }
      const float2 a = __ffma2_rn(make_float2(x[e], x[e + 1]), cc, nm);
      pk[i] = pack_bf16(ex2(a.x), ex2(a.y));
    }
    if (__any_sync(0xffffffffu, fmaxf(m0, m1) * c > m + kRescaleLog2)) {
      softmax_tile_redo(tS, tO, c, m, la, lb);
      return;
    }
    tmem_st32(tS, pk);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i & 1) add_bf16x2_f32(lb, pk[i]); else add_bf16x2_f32(la, pk[i]);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = 64 + 2 * i;
      const float2 a = __ffma2_rn(make_float2(x[e], x[e + 1]), cc, nm);
      pk[i] = pack_bf16(ex2(a.x), ex2(a.y));
      if (i & 1) add_bf16x2_f32(lb, pk[i]); else add_bf16x2_f32(la, pk[i]);
    }
    tmem_st32(tS + 32, pk);
    return;
  }
  float mx;
  if (kFull) {
    // columns 0-3 seed four chains, 4-123 take 15 rounds of 8, 124-127 close two chains
    float m0 = x[0], m1 = x[1], m2 = x[2], m3 = x[3];
#pragma unroll
    for (int i = 4; i < 124; i += 8) {
      m0 = fmax3(m0, x[i], x[i + 1]);
      m1 = fmax3(m1, x[i + 2], x[i + 3]);
      m2 = fmax3(m2, x[i + 4], x[i + 5]);
      m3 = fmax3(m3, x[i + 6], x[i + 7]);
    }
    m0 = fmax3(m0, x[124], x[125]);
    m1 = fmax3(m1, x[126], x[127]);
    mx = fmax3(m0, m1, fmaxf(m2, m3));
  } else {
    mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 128; ++i)
      if (i < kv_valid) mx = fmaxf(mx, x[i]);
  }
  const float m_new = fmaxf(m, mx * c);
  if (first) {
    m = m_new;
  } else if (__any_sync(0xffffffffu, m_new > m + kRescaleLog2)) {
    const float alpha = ex2(m - m_new);
    la = __fmul2_rn(la, make_float2(alpha, alpha));
    lb = __fmul2_rn(lb, make_float2(alpha, alpha));
    m = m_new;
#pragma unroll 1
    for (int h = 0; h < 4; ++h) {
      float o[32];
      tmem_ld32(tO + 32 * h, o);
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(o[i] * alpha);
      tmem_st32(tO + 32 * h, r);
    }
    tmem_wait_st();
    // Rare path: the scores are read again instead of being kept live across
    // the rescale, which keeps the register budget of the common path.
    tmem_ld128(tS, x);
  }
  const float2 cc = make_float2(c, c);
  const float2 nm = make_float2(-m, -m);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = 64 * h + 2 * i;
      const float2 a = __ffma2_rn(make_float2(x[e], x[e + 1]), cc, nm);
      float p0 = ex2(a.x), p1 = ex2(a.y);
      if (!kFull) {
        p0 = e < kv_valid ? p0 : 0.f;
        p1 = e + 1 < kv_valid ? p1 : 0.f;
      }
      pk[i] = pack_bf16(p0, p1);
      // The row sum uses the bf16-rounded P that the P V product sees, so the
      // output is an exact convex combination of V rows up to fp32
      // accumulation (matters for peaked rows where |O| approaches |V|).
      if (i & 1) add_bf16x2_f32(lb, pk[i]); else add_bf16x2_f32(la, pk[i]);
    }
    // P (bf16 pairs): S columns 64h..64h+63 become P columns 32h..32h+31.
    tmem_st32(tS + 32 * h, pk);
  }
}

// Softmax warps: warp w handles Q tile w/4, TMEM lanes 32*(w%4) .. +31; the
// thread owns one query row.
template <bool kText, bool kSpec>
__device__ __forceinline__ void softmax_role(const TcParams& prm, const Smem& sm, uint32_t tmem, int warp,
                                             int lane) {
  int* err = prm.work + WS_ERROR;
  const int t = warp >> 2;
  const int rq = (warp & 3) * 32 + lane;
  const uint32_t lane_bits = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_bits + (t ? kColS1 : kColS0);
  const uint32_t tO = tmem + lane_bits + (t ? kColO1 : kColO0);
  const float c = prm.c;
  uint32_t unit_iter = 0, s_iter = 0, o_iter = 0;
  while (true) {
    const int us = unit_iter & 1;
    if (!__all_sync(0xffffffffu, wait_bar(bar_at(sm, B_UNIT_FULL + us), (unit_iter >> 1) & 1, err, E_SM_UNIT_FULL)))
      break;
    const int4 info = sm.units[us];
    if (info.y < 0) break;
    const int off = info.x, nv = info.y, q0 = info.z, head = info.w & 0xffff;
    const int nvt = (nv + kTile - 1) / kTile;
    const int nkv = nvt + (kText ? (prm.n_text + kTile - 1) / kTile : 0);
    const int qtile = q0 / kTile + t;
    if (qtile < nkv) {
      float m = -INFINITY;
      float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        ok = __all_sync(0xffffffffu, wait_bar(bar_at(sm, B_S_FULL + t), s_iter & 1, err, E_SM_S_FULL));
        ++s_iter;
        if (!ok) break;
        tc_fence_after();
        const int kv_valid =
            !kText || j < nvt ? min(kTile, nv - j * kTile) : min(kTile, prm.n_text - (j - nvt) * kTile);
        if (kv_valid == kTile)
          softmax_tile<true, kSpec>(tS, tO, j == 0, kv_valid, c, m, la, lb);
        else
          softmax_tile<false, kSpec>(tS, tO, j == 0, kv_valid, c, m, la, lb);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_at(sm, B_P_FULL + t));
      }
      if (!ok) break;
      if (!__all_sync(0xffffffffu, wait_bar(bar_at(sm, B_O_FULL + t), o_iter & 1, err, E_SM_O_FULL))) break;
      ++o_iter;
      tc_fence_after();
      const float inv = 1.f / ((la.x + la.y) + (lb.x + lb.y));
      const bool vtile = !kText || qtile < nvt;
      const int qr = (vtile ? qtile : qtile - nvt) * kTile + rq;  // row of the video or the text part
      bool valid = vtile && qr < nv;                                // a video row of this window
      const bool text = kText && !vtile && qr < prm.n_text;         // a text row: partial T_w / W
      long long tok = 0;
      if (valid) tok = prm.row_map ? __ldg(prm.row_map + off + qr) : off + qr;
      if (kBoundsCheck && valid && static_cast<unsigned long long>(tok) >= static_cast<unsigned long long>(prm.n_tokens)) {
        atomicCAS(prm.work + WS_BOUNDS, 0, kErrBounds);
        valid = false;  // not written
        tok = 0;
      }
      float* tdst = nullptr;
      if (text) {
        const long long window = static_cast<unsigned>(info.w) >> 16;
        tdst = prm.text_part + ((window * prm.n_text + qr) * prm.heads + head) * kD;
      }
      uint4* dst = reinterpret_cast<uint4*>(prm.o + tok * prm.row_stride + static_cast<long long>(head) * (kD * 2));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float x[64];
        __syncwarp();
        tmem_ld64(tO + 64 * h, x);
        if (kText && text) {
          const float sc = inv * prm.inv_windows;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            st_global_v8(tdst + 64 * h + 8 * k, __float_as_uint(x[8 * k] * sc), __float_as_uint(x[8 * k + 1] * sc),
                         __float_as_uint(x[8 * k + 2] * sc), __float_as_uint(x[8 * k + 3] * sc),
                         __float_as_uint(x[8 * k + 4] * sc), __float_as_uint(x[8 * k + 5] * sc),
                         __float_as_uint(x[8 * k + 6] * sc), __float_as_uint(x[8 * k + 7] * sc));
        }
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(x[2 * i] * inv, x[2 * i + 1] * inv);
        if (valid) {
          if (prm.o_v8) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              st_global_v8(dst + 8 * h + 2 * k, pk[8 * k], pk[8 * k + 1], pk[8 * k + 2], pk[8 * k + 3], pk[8 * k + 4],
                           pk[8 * k + 5], pk[8 * k + 6], pk[8 * k + 7]);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              st_global_v4(dst + 8 * h + k, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          }
        }
      }
      tc_fence_before();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_at(sm, B_UNIT_EMPTY + us));
    ++unit_iter;
  }
}

// Registers: each SM sub-partition holds 16K registers and 3 of the 12
// warps, so 168 registers per thread fit (3 x 32 x 168 = 16,128).
template <bool kText, bool kTma>
__global__ void __maxnreg__(168) attention_tc_kernel(const __grid_constant__ TcParams prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  Smem sm;
  sm.q0 = base + kSmemQ;
  sm.ring = base + kSmemRing;
  sm.bars = base + kSmemBars;
  sm.units = reinterpret_cast<int4*>(base_ptr + kSmemUnits);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + kSmemTmem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar_at(sm, B_RING_FULL + s), 32 * kLoaderWarps);
      mbar_init(bar_at(sm, B_RING_EMPTY + s), 1);
    }
    mbar_init(bar_at(sm, B_Q_FULL), 32 * kLoaderWarps);
    mbar_init(bar_at(sm, B_Q_EMPTY), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_at(sm, B_S_FULL + t), 1);
      mbar_init(bar_at(sm, B_P_FULL + t), 128);
      mbar_init(bar_at(sm, B_O_FULL + t), 1);
      mbar_init(bar_at(sm, B_UNIT_FULL + t), 1);
      mbar_init(bar_at(sm, B_UNIT_EMPTY + t), kLoaderWarps + 1 + 8);
    }
    mbar_init(bar_at(sm, B_DRAIN), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp < kLoaderWarp0) {
    softmax_role<kText, kTma>(prm, sm, tmem, warp, lane);
  } else if (warp < kMmaWarp) {
    loader_role<kText, kTma>(prm, sm, warp - kLoaderWarp0, lane);
  } else if (warp == kMmaWarp) {
    mma_role<kText>(prm, sm, tmem);
  } else if (lane == 0) {
    scheduler_role(prm, sm);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // The last CTA to finish resets the scheduler for the next launch.
    __threadfence();
    const int prev = atomicAdd(prm.work + WS_DONE_CTAS, 1);
    if (prev == static_cast<int>(gridDim.x) - 1) {
      atomicExch(prm.work + WS_NEXT_UNIT, 0);
      atomicExch(prm.work + WS_DONE_CTAS, 0);
      __threadfence();
    }
  }
}

}  // namespace

namespace {

// Text output: o_txt[t][c] = sum over windows w of part[w][t][c] (each
// partial already divided by the window count), summed in window order so
// the result does not depend on scheduling; converted to bf16.
__global__ void text_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ out, long long per_window,
                                   int windows) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < per_window;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float acc = 0.f;
    for (int w = 0; w < windows; ++w) acc += part[w * per_window + i];
    out[i] = __float2bfloat16_rn(acc);
  }
}

}  // namespace

namespace {

// Rows of a text segment as the kernel tiles it: the video part and the text
// part each padded to whole 128-row tiles.
int text_segment_rows(int nv, int n_text) { return ((nv + 127) / 128 + (n_text + 127) / 128) * 128; }

}  // namespace

size_t attention_text_workspace_bytes(const wsa_plan_s& p, int n_text, int heads, size_t* items_bytes) {
  std::vector<int> seg(p.h_offsets.size(), 0);
  for (size_t w = 1; w < seg.size(); ++w)
    seg[w] = seg[w - 1] + text_segment_rows(p.h_offsets[w] - p.h_offsets[w - 1], n_text);
  const size_t n_items = make_items(seg, kTcItemRows, 128).size();
  const size_t ib = (n_items * sizeof(WorkItem) + 255) / 256 * 256;
  if (items_bytes) *items_bytes = ib;
  return ib + static_cast<size_t>(p.num_windows) * n_text * heads * kD * sizeof(float);
}

cudaError_t launch_attention_text_bf16_tc(const wsa_plan_s& p, const void* q, const void* k, const void* v, void* o,
                                          const void* qt, const void* kt, const void* vt, void* ot, int n_text,
                                          int heads, bool canonical, float scale, void* workspace, cudaStream_t s) {
  std::vector<int> seg(p.h_offsets.size(), 0);
  for (size_t w = 1; w < seg.size(); ++w)
    seg[w] = seg[w - 1] + text_segment_rows(p.h_offsets[w] - p.h_offsets[w - 1], n_text);
  const std::vector<WorkItem> items = make_items(seg, kTcItemRows, 128);
  size_t items_bytes = 0;
  attention_text_workspace_bytes(p, n_text, heads, &items_bytes);
  WorkItem* d_items = static_cast<WorkItem*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + items_bytes);
  // pageable source: the copy stages the vector before returning
  cudaError_t e = cudaMemcpyAsync(d_items, items.data(), items.size() * sizeof(WorkItem), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  e = launch_attention_tc(p, q, k, v, o, heads, canonical, scale, s, qt, kt, vt, part, n_text, d_items,
                          static_cast<int>(items.size()));
  if (e != cudaSuccess) return e;
  const long long per_window = static_cast<long long>(n_text) * heads * kD;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<long long>((per_window + threads - 1) / threads, 8LL * sm_count()));
  text_reduce_kernel<<<std::max(1, blocks), threads, 0, s>>>(part, static_cast<__nv_bfloat16*>(ot), per_window,
                                                              p.num_windows);
  return cudaGetLastError();
}

cudaError_t launch_attention_bf16_tc(const wsa_plan_s& p, const void* q, const void* k, const void* v, void* o,
                                     int heads, bool canonical, float scale, cudaStream_t s) {
  return launch_attention_tc(p, q, k, v, o, heads, canonical, scale, s, nullptr, nullptr, nullptr, nullptr, 0,
                             p.d_tc_items, p.num_tc_items);
}

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library itself); null if unavailable.
EncodeTiled encoder() {
  static const EncodeTiled fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiled>(nullptr);
    return reinterpret_cast<EncodeTiled>(f);
  }();
  return fn;
}

// Tile map of a [rows, heads, 128] bf16 tensor: box of 64 channels x 1 head x
// 128 rows, 128-byte swizzle, rows past the end read as zero.
cudaError_t encode_rows(CUtensorMap* map, const void* base, int rows, int heads) {
  const EncodeTiled enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(heads) * kD * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kTile)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

namespace {
std::atomic<int> g_withhold_launches{0};
}  // namespace

void withhold_attention_units(int launches) { g_withhold_launches.store(launches < 0 ? 0 : launches); }

cudaError_t launch_attention_tc(const wsa_plan_s& p, const void* q, const void* k, const void* v, void* o, int heads,
                                bool canonical, float scale, cudaStream_t s, const void* qt, const void* kt,
                                const void* vt, float* text_part, int n_text, const WorkItem* items, int n_items) {
  TcParams prm;
  std::memset(&prm, 0, sizeof(prm));
  for (int n = g_withhold_launches.load(); n > 0;) {
    if (g_withhold_launches.compare_exchange_weak(n, n - 1)) {
      prm.withhold_units = 1;
      break;
    }
  }
  // Packed rows without a text segment: full tiles by TMA.
  const bool tma = !canonical && n_text == 0;
  if (tma) {
    cudaError_t e = encode_rows(&prm.tm_q, q, p.num_tokens, heads);
    if (e == cudaSuccess) e = encode_rows(&prm.tm_k, k, p.num_tokens, heads);
    if (e == cudaSuccess) e = encode_rows(&prm.tm_v, v, p.num_tokens, heads);
    if (e != cudaSuccess) return e;
  }
  prm.q = static_cast<const char*>(q);
  prm.k = static_cast<const char*>(k);
  prm.v = static_cast<const char*>(v);
  prm.o = static_cast<char*>(o);
  prm.row_map = canonical ? p.d_ids : nullptr;
  prm.offsets = p.d_offsets;
  prm.items = items;
  prm.num_units = n_items * heads;
  prm.qt = static_cast<const char*>(qt);
  prm.kt = static_cast<const char*>(kt);
  prm.vt = static_cast<const char*>(vt);
  prm.text_part = text_part;
  prm.n_text = n_text;
  prm.inv_windows = 1.0f / static_cast<float>(p.num_windows);
  prm.heads = heads;
  prm.n_tokens = p.num_tokens;
  prm.row_stride = static_cast<long long>(heads) * kD * 2;
  prm.c = scale * 1.4426950408889634f;
  prm.o_v8 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 && (prm.row_stride & 31) == 0;
  prm.work = p.d_work;
  // The text segment is a separate instantiation: its extra row source costs
  // the video-only kernel's gather warps issue slots even where it never runs.
  auto kernel = n_text > 0 ? attention_tc_kernel<true, false>
                           : (tma ? attention_tc_kernel<false, true> : attention_tc_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(sm_count(), prm.num_units));
  kernel<<<grid, kThreads, kSmemAlloc, s>>>(prm);
  return cudaGetLastError();
}

}  // namespace wsa
