// Tensor-core GEMMs for sm_103a: D = alpha * A B^T (+ bias), A [M, K] and B [N, K]
// contraction-major, fp32 accumulation in tensor memory (TMEM).
//
// One persistent kernel template serves the four operand kinds:
//   BF16   tcgen05.mma kind::f16              K = 16 per instruction
//   FP8    tcgen05.mma kind::f8f6f4           K = 32, per-tensor alpha in the epilogue
//   MXFP8  tcgen05.mma kind::mxf8f6f4         K = 32, E8M0 scale per 32 elements (block_scale 1X)
//   NVFP4  tcgen05.mma kind::mxf4nvf4         K = 64, UE4M3 scale per 16 elements (block_scale 4X)
// Every kind moves 32 bytes of each operand row per instruction, so one k-tile
// is a 128-byte row slice (one 128-byte-swizzle atom) and 4 instructions.
//
// CTA = 10 warps (MXFP8 11, NVFP4 12), one CTA per SM (the shared-memory footprint guarantees it):
//   warp 0      TMA producer: A tile [128 x 128 B], B tile and, for the block-scaled
//               kinds, the scale-factor atoms, into a shared-memory ring guarded by
//               full/empty mbarriers;
//   warp 1      allocates TMEM and issues the MMAs from one thread (for block-scaled
//               kinds once the stage's scale factors are in TMEM): each k-tile's MMAs
//               are followed by tcgen05.commit onto the stage's empty barrier, each
//               tile's last k-tile by a commit onto the accumulator-full barrier;
//   warps 2-9   epilogue: each warp owns a 32-lane quarter of TMEM and a 128-column
//               half of the 128 x 256 accumulator, drains it to registers, releases
//               the accumulator, then applies alpha / bias, rounds and stores;
//   warp 10(-11) block-scaled kinds: issue the scale-factor copies (NVFP4 12, MXFP8 3 per
//               k-tile) as soon as a stage lands and commit them onto the stage's
//               sf_ready barrier, so they run beside the MMAs of earlier k-tiles (copies
//               and MMAs from one thread execute in issue order).  One thread's copies
//               complete at about one per 46 ns, so NVFP4 splits its 12 between two warps.
// Every kind runs as CTA pairs (2-CTA clusters, tcgen05 cta_group::2) on 256 x 256
// tiles: each CTA stages 128 rows of A and 128 rows of B (BF16 / FP8 / MXFP8 6 stages,
// NVFP4 5), the leader's thread issues M = 256 MMAs that read both CTAs' operands and
// write each CTA's 128 accumulator rows into its own TMEM, and its commits free the
// stage and publish the accumulator in both CTAs; loads of both CTAs complete on the
// leader's full barrier, and both CTAs' epilogue warps arrive on the leader's
// accumulator-empty barrier.  Halving each SM's share of B halves its shared-memory
// traffic for B.  Block-scaled kinds: each half of a pair MMA reads every B row's
// scales from its own TMEM, so each CTA stages the scale atoms of all 256 B rows (and
// its own 128 A rows); the pair tcgen05.cp copies each CTA's own shared memory into
// its own TMEM; the atoms arrive by TMA so that they complete on the leader's barrier.
// (The template also builds one CTA per 128 x 256 tile, CG = 1; no entry point uses it.)
// The accumulator is double-buffered in TMEM for BF16/FP8 (2 x 256 columns); the
// block-scaled kinds keep one 256-column accumulator plus a per-stage scale-factor
// region and rely on the early release of the register drain for overlap.
// Tiles are visited in a grouped raster (16 pair M-tiles, 4096 rows, per group) so
// concurrently running CTAs share A and B tiles in L2, and B is streamed from DRAM
// once per group (8-bit kinds on long contractions: the smaller operand's tiles fastest);
// each CTA walks K forwards on its even tiles and backwards on its odd ones, so that
// consecutive waves of tiles meet in L2.  No cluster multicast is used.
#include <cuda_bf16.h>

#include "common.cuh"

namespace te {
namespace {

enum Kind { kBF16 = 0, kFP8 = 1, kMXFP8 = 2, kNVFP4 = 3 };

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kEpiWarps = 8;
constexpr int kCopyWarp = 2 + kEpiWarps;               // first scale-factor copier (block-scaled kinds)
constexpr int kGroupM = 16;

// CG = 1: one CTA per 128 x 256 tile.  CG = 2 (BF16 / FP8): a CTA pair per 256 x 256
// tile with the pair-wide MMA (tcgen05 cta_group::2): each CTA holds 128 rows of A
// and 128 rows of B, the leader's single thread issues M = 256 MMAs that read both
// CTAs' shared memory and write each CTA's own 128 accumulator rows in its TMEM.
template <int KIND, int CG = 1>
struct Cfg {
  static constexpr bool kPair = CG == 2;
  static constexpr int kBRows = BN / CG;                      // B rows staged by one CTA
  static constexpr int kStages = kPair ? (KIND == kNVFP4 ? 5 : 6) : (KIND == kNVFP4 ? 3 : 4);
  static constexpr bool kBlockScaled = KIND >= kMXFP8;
  static constexpr int kAccStages = kBlockScaled ? 1 : 2;
  // The scale copies (NVFP4 12, MXFP8 3 per k-tile) go out from copier warps of their own,
  // so the tensor pipe overlaps them with the MMAs (pairs: NVFP4 +12 %, MXFP8 +11 %).  One
  // thread's copies complete at about one per 46 ns whatever their size, so NVFP4's 12 per
  // k-tile from one thread outlast the k-tile's MMAs: two copier warps, each issuing the
  // copies of half the k-steps (+29 %).  BF16 and FP8 have no scales and no copier warp.
  static constexpr int kSfCopiers = KIND == kNVFP4 ? 2 : (kBlockScaled ? 1 : 0);
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kSfCopiers);
  static constexpr uint32_t kTmemCols = 512u;
  static constexpr int kABytes = BM * 128;
  static constexpr int kBBytes = kBRows * 128;
  // scale-factor atoms (512 B = 128 rows x 4 scales) per 128 rows per k-tile
  static constexpr int kSfAtoms = KIND == kMXFP8 ? 1 : (KIND == kNVFP4 ? 4 : 0);
  static constexpr int kSfaBytes = kSfAtoms * 512;
  // B's scale atoms of all 256 B rows per k-tile: in a pair each CTA's half of the MMA
  // reads the scales of every B row from its own TMEM
  static constexpr int kSfbAtoms = 2 * kSfAtoms;
  static constexpr int kSfbBytes = kSfbAtoms * 512;
  static constexpr int kSfaCols = 4 * kSfAtoms;
  static constexpr int kSfbCols = 4 * kSfbAtoms;
  static constexpr int kSfTmemBase = 256;
  static constexpr int kSmemA = 0;
  static constexpr int kSmemB = kSmemA + kStages * kABytes;
  static constexpr int kSmemSfa = kSmemB + kStages * kBBytes;
  static constexpr int kSmemSfb = kSmemSfa + kStages * kSfaBytes;
  static constexpr int kSmemStage = kSmemSfb + kStages * kSfbBytes;      // epilogue staging, 2 KB per warp
  static constexpr int kSmemBar = kSmemStage + kEpiWarps * 2048;
  static constexpr int kSmemTotal = kSmemBar + 256 + 1024;  // barriers + alignment slack
  static_assert((4 * kStages + 5) * 8 + 8 <= 256, "barrier area");
  static_assert(!kBlockScaled || kSfTmemBase + kStages * (kSfaCols + kSfbCols) <= int(kTmemCols), "TMEM budget");
  static_assert(kSmemTotal <= 232448, "shared memory budget");
};

struct GemmArgs {
  int M, N, K;
  int k_tiles, m_tiles, n_tiles;
  const uint8_t* sfa;
  const uint8_t* sfb;
  int64_t sf_katoms;    // scale atoms per 128-row group (padded scale columns / 4)
  int sfb_row_atoms;    // 128-row groups present in B's scale tensor
  const float* alpha_a;
  const float* alpha_b;
  const float* bias;
  void* D;
  int out_f32;
  int accumulate;       // 1: D (fp32) += result, by TMA reduce-add
  uint32_t idesc;
  int a_mn, b_mn;       // BF16 only: operand stored [K, M] / [K, N]
  int raster;           // 1: the smaller operand's tiles vary fastest (see tile_coords)
  int* err;
};

// Tile `tile` of the persistent walk -> (M tile, N tile).  Grouped raster: 16 pair M-tiles at
// a time, M fastest.  raster = 1 (8-bit kinds on long contractions): the smaller operand's tiles
// vary fastest, so each wave sweeps all of it and it stays in L2 across waves while the other
// streams once (FP8 DRAM traffic 1.74 -> 1.52 x the operands over the layer's 12 GEMMs, 0.4 %
// faster; on the K = 4096 shapes, and for BF16, it cost time).
__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int& mt, int& nt, int raster = 0) {
  if (raster) {
    if (m_tiles >= n_tiles) mt = tile / n_tiles, nt = tile % n_tiles;
    else mt = tile % m_tiles, nt = tile / m_tiles;
    return;
  }
  const int group = kGroupM * n_tiles;
  const int g = tile / group;
  const int first_m = g * kGroupM;
  const int gm = min(m_tiles - first_m, kGroupM);
  const int in_group = tile - g * group;
  mt = first_m + in_group % gm;
  nt = in_group / gm;
}

template <int KIND, int CG>
__global__ void __launch_bounds__(Cfg<KIND, CG>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmSa,
                const __grid_constant__ CUtensorMap tmSb, const __grid_constant__ GemmArgs args) {
  using C = Cfg<KIND, CG>;
  constexpr bool kPair = C::kPair;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = dev::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sA = smem + C::kSmemA;
  uint8_t* sB = smem + C::kSmemB;
  uint8_t* sSfa = smem + C::kSmemSfa;
  uint8_t* sSfb = smem + C::kSmemSfb;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kSmemBar);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* sf_ready = drain + 1;  // [kStages]: the stage's scale factors are in TMEM
  uint64_t* sf_full = sf_ready + kStages;   // [kStages]: the stage's scale atoms have landed (block-scaled kinds)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = args.m_tiles * args.n_tiles;   // m_tiles counts BM * CG rows
  // CTA pairs: rank 0 (the leader) issues the MMAs; both CTAs load, drain and store.
  const uint32_t rank = kPair ? dev::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      dev::mbar_init(&acc_full[s], 1);
      dev::mbar_init(&acc_empty[s], CG * kEpiWarps);   // one arrival per epilogue warp of each CTA
    }
    dev::mbar_init(drain, 1);
    for (int st = 0; st < kStages; ++st) {
      dev::mbar_init(&sf_ready[st], C::kSfCopiers > 0 ? C::kSfCopiers : 1);
      dev::mbar_init(&sf_full[st], 1);
    }
    *abort_flag = 0;
    dev::fence_barrier_init();
    dev::prefetch_tmap(&tmA);
    dev::prefetch_tmap(&tmB);
    dev::prefetch_tmap(&tmD);
  }
  if (kPair) dev::cluster_sync();  // the peer's barriers are initialised before anyone signals them
  if (warp == 1) {
    if (kPair) dev::tmem_alloc_pair(tmem_slot, C::kTmemCols);
    else dev::tmem_alloc(tmem_slot, C::kTmemCols);
  }
  dev::tc_fence_before();
  __syncthreads();
  if (kPair) dev::cluster_sync();
  dev::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (kPair && !leader && threadIdx.x == 0) {
    // the pair-wide allocation hands both CTAs the same columns; anything else is unusable
    if (dev::ld_shared_cluster_u32(dev::mapa_shared(dev::smem_u32(tmem_slot), 0)) != tmem_base) {
      dev::set_error(args.err, TE_ERR_UNSUPPORTED);
      *abort_flag = 1;
    }
  }
  __syncthreads();

  // Scale atoms j = j0, j0 + dj, ... of stage `st` (shared memory) -> its TMEM slot, one copy
  // per 512-byte atom, the A atom and the two B atoms of a k-step back to back (grouped by
  // k-step the copies run 15-30 % faster than grouped by operand).
  auto issue_sf_copies = [&](int st, int j0, int dj) {
    const uint32_t sfa_t = tmem_base + C::kSfTmemBase + static_cast<uint32_t>(st * (C::kSfaCols + C::kSfbCols));
    const uint32_t sfb_t = sfa_t + C::kSfaCols;
    const uint32_t sfa_s = dev::smem_u32(sSfa + st * C::kSfaBytes);
    const uint32_t sfb_s = dev::smem_u32(sSfb + st * C::kSfbBytes);
    auto cp = [&](uint32_t t, uint32_t sa) {
      if (kPair) dev::tc_cp_32x128b_x4_pair(t, dev::smem_desc(sa, 0, 128, 0));
      else dev::tc_cp_32x128b_x4(t, dev::smem_desc(sa, 0, 128, 0));
    };
#pragma unroll
    for (int j = 0; j < C::kSfAtoms; ++j) {
      if (j < j0 || (j - j0) % dj != 0) continue;
      cp(sfa_t + 4 * j, sfa_s + 512 * j);
#pragma unroll
      for (int h = 0; h < 2; ++h) cp(sfb_t + 8 * j + 4 * h, sfb_s + h * C::kSfAtoms * 512 + 512 * j);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[kStages];
      bool issued[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = false, issued_phase[s] = 0;
      // pairs: the leader's barriers count both CTAs' bytes.  Block-scaled kinds: the scale
      // atoms are loaded first and land on their own barrier (sf_full), so the copier warps
      // move them into TMEM while the stage's operand tiles are still arriving.
      const uint32_t tx = kPair ? (C::kABytes + C::kBBytes) * CG : C::kABytes + C::kBBytes;
      const uint32_t sf_tx0 = kPair ? (C::kSfaBytes + C::kSfbBytes) * CG : C::kSfaBytes;
      bool ok = !*abort_flag;
      int it = 0;
      for (int tile = unit; tile < num_tiles && ok; tile += units, ++it) {
        int mt, nt;
        tile_coords(tile, args.m_tiles, args.n_tiles, mt, nt, args.raster);
        for (int kt0 = 0; kt0 < args.k_tiles; ++kt0) {
          // Every other tile of a CTA walks K backwards: the CTAs run their tiles in waves,
          // and a wave that starts where the previous one ended finds the panels' last
          // k-slices still in L2 (FP8, 12 layer shapes: DRAM traffic 2.16 -> 1.72 x the
          // operands, 1-2 % faster).  Only the order of the fp32 partial sums changes.
          const int kt = (it & 1) ? args.k_tiles - 1 - kt0 : kt0;
          if (!dev::mbar_wait<kPair>(&empty[stage], phase ^ 1u, abort_flag, args.err)) {
            ok = false;
            break;
          }
          uint32_t sf_tx = sf_tx0;
          if (C::kBlockScaled && !kPair) {
            for (int h = 0; h < 2; ++h)
              if (nt * 2 + h < args.sfb_row_atoms) sf_tx += C::kSfAtoms * 512;
          }
          if (leader) {
            if (C::kBlockScaled) dev::mbar_expect_tx(&sf_full[stage], sf_tx);
            dev::mbar_expect_tx(&full[stage], tx);
          }
          const int arow = (mt * CG + static_cast<int>(rank)) * BM;         // this CTA's A rows
          const int brow = nt * BN + static_cast<int>(rank) * C::kBRows;    // this CTA's B rows
          const uint32_t full_c = dev::mapa_shared(dev::smem_u32(&full[stage]), 0);
          const uint32_t sf_full_c = dev::mapa_shared(dev::smem_u32(&sf_full[stage]), 0);
          auto load = [&](uint8_t* dst, const CUtensorMap* map, int x, int y) {
            if (kPair) dev::tma_load_2d_pair(dst, map, full_c, x, y);
            else dev::tma_load_2d(dst, map, &full[stage], x, y);
          };
          auto load_sf = [&](uint8_t* dst, const CUtensorMap* map, int x, int y) {
            if (kPair) dev::tma_load_2d_pair(dst, map, sf_full_c, x, y);
          };
          if (C::kBlockScaled && kPair) {
            // scale atoms by TMA, first (completion on the leader's sf_full barrier): the scale
            // tensor is viewed as 256-byte rows, so a 128-row group's atoms of one k-tile are
            // 2 * kSfAtoms consecutive rows; boxes past the end are zero-filled
            const int64_t katom = static_cast<int64_t>(kt) * C::kSfAtoms;
            load_sf(sSfa + stage * C::kSfaBytes, &tmSa, 0,
                    static_cast<int>(((mt * CG + static_cast<int>(rank)) * args.sf_katoms + katom) * 2));
            for (int h = 0; h < 2; ++h)
              load_sf(sSfb + stage * C::kSfbBytes + h * C::kSfAtoms * 512, &tmSb, 0,
                      static_cast<int>(((nt * 2 + h) * args.sf_katoms + katom) * 2));
          } else if (C::kBlockScaled) {
            const int64_t katom = static_cast<int64_t>(kt) * C::kSfAtoms;
            dev::bulk_load(sSfa + stage * C::kSfaBytes, args.sfa + (mt * args.sf_katoms + katom) * 512,
                           C::kSfaBytes, &sf_full[stage]);
            for (int h = 0; h < 2; ++h) {
              const int ra = nt * 2 + h;
              if (ra < args.sfb_row_atoms)
                dev::bulk_load(sSfb + stage * C::kSfbBytes + h * C::kSfAtoms * 512,
                               args.sfb + (ra * args.sf_katoms + katom) * 512, C::kSfAtoms * 512, &sf_full[stage]);
            }
          }
          if (KIND == kBF16 && args.a_mn) {
            // [K, M] storage: 64 K-rows x 64 M-elements (128 B) per box, two boxes along M
#pragma unroll
            for (int h = 0; h < BM / 64; ++h) load(sA + stage * C::kABytes + h * 8192, &tmA, (arow + 64 * h) * 2, kt * 64);
          } else {
            load(sA + stage * C::kABytes, &tmA, kt * 128, arow);
          }
          if (KIND == kBF16 && args.b_mn) {
#pragma unroll
            for (int h = 0; h < C::kBRows / 64; ++h)
              load(sB + stage * C::kBBytes + h * 8192, &tmB, (brow + 64 * h) * 2, kt * 64);
          } else {
            load(sB + stage * C::kBBytes, &tmB, kt * 128, brow);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
      }
      if (!ok && leader) {
        // Bounded wait for copies still in flight before the CTA exits (a pair's leader
        // barrier also counts the peer's copies; the peer cannot leave before the
        // leader, whose exit waits on the final cluster barrier).
        volatile int dummy = 0;
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) {
            dev::mbar_wait(&full[s], issued_phase[s], &dummy, args.err);
            if (C::kBlockScaled) dev::mbar_wait(&sf_full[s], issued_phase[s], &dummy, args.err);
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (one thread; the pair's leader)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = !*abort_flag;
      auto commit = [&](uint64_t* bar, uint16_t mask) {
        if (kPair) dev::tc_commit_pair(bar, mask);
        else dev::tc_commit(bar);
      };
      auto sf_slot = [&](int st) {
        return tmem_base + C::kSfTmemBase + static_cast<uint32_t>(st * (C::kSfaCols + C::kSfbCols));
      };
      for (int tile = unit; tile < num_tiles && ok; tile += units, ++it) {
        const int as = it % C::kAccStages;
        const uint32_t aphase = static_cast<uint32_t>(it / C::kAccStages) & 1u;
        if (!dev::mbar_wait<kPair>(&acc_empty[as], aphase ^ 1u, abort_flag, args.err)) {
          ok = false;
          break;
        }
        dev::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as * BN);
        for (int kt = 0; kt < args.k_tiles; ++kt) {
          const int nstage = stage + 1 == kStages ? 0 : stage + 1;
          const uint32_t nphase = stage + 1 == kStages ? phase ^ 1u : phase;
          const uint32_t a_addr = dev::smem_u32(sA + stage * C::kABytes);
          const uint32_t b_addr = dev::smem_u32(sB + stage * C::kBBytes);
          const uint32_t sfa_t = sf_slot(stage), sfb_t = sfa_t + C::kSfaCols;
          // the stage's addresses first, so that little stands between a barrier's completion
          // and the first MMA (MXFP8 1 % faster); the scale factors of this k-tile reach the
          // stage's TMEM slot from the copier warps, whose copies run beside this thread's
          // MMAs of earlier k-tiles
          if (!dev::mbar_wait<kPair>(&full[stage], phase, abort_flag, args.err)) {
            ok = false;
            break;
          }
          if (C::kBlockScaled && !dev::mbar_wait<kPair>(&sf_ready[stage], phase, abort_flag, args.err)) {
            ok = false;
            break;
          }
          dev::tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            // K-major: 128-byte rows, 8-row swizzle atoms 1024 B apart; a k-step advances 32 B.
            // MN-major (BF16): 64-element x 8-K-row atoms, 1024 B apart along K (SBO) and
            // 8 KB apart along M / N (LBO); a k-step of 16 K-rows advances 2048 B.
            const uint64_t adesc = (KIND == kBF16 && args.a_mn) ? dev::smem_desc(a_addr + 2048 * ks, 8192, 1024, 2)
                                                                : dev::smem_desc(a_addr + 32 * ks, 0, 1024, 2);
            const uint64_t bdesc = (KIND == kBF16 && args.b_mn) ? dev::smem_desc(b_addr + 2048 * ks, 8192, 1024, 2)
                                                                : dev::smem_desc(b_addr + 32 * ks, 0, 1024, 2);
            const uint32_t acc = (kt | ks) != 0;
            if (KIND == kBF16) {
              if (kPair) dev::mma_f16_pair(d_tmem, adesc, bdesc, args.idesc, acc);
              else dev::mma_f16(d_tmem, adesc, bdesc, args.idesc, acc);
            } else if (KIND == kFP8) {
              if (kPair) dev::mma_f8f6f4_pair(d_tmem, adesc, bdesc, args.idesc, acc);
              else dev::mma_f8f6f4(d_tmem, adesc, bdesc, args.idesc, acc);
            } else if (KIND == kMXFP8) {
              // scale byte `ks` of each 32-bit scale column (bits 29-30: A, bits 4-5: B)
              const uint32_t idesc = args.idesc | (static_cast<uint32_t>(ks) << 29) | (static_cast<uint32_t>(ks) << 4);
              if (kPair) dev::mma_mxf8f6f4_pair(d_tmem, adesc, bdesc, idesc, sfa_t, sfb_t, acc);
              else dev::mma_mxf8f6f4(d_tmem, adesc, bdesc, idesc, sfa_t, sfb_t, acc);
            } else {
              const uint32_t sfb_k = sfb_t + 8 * ks;
              if (kPair) dev::mma_mxf4nvf4_pair(d_tmem, adesc, bdesc, args.idesc, sfa_t + 4 * ks, sfb_k, acc);
              else dev::mma_mxf4nvf4(d_tmem, adesc, bdesc, args.idesc, sfa_t + 4 * ks, sfb_k, acc);
            }
          }
          commit(&empty[stage], 3);   // frees the stage in both CTAs of a pair
          stage = nstage;
          phase = nphase;
        }
        if (!ok) break;
        commit(&acc_full[as], 3);
      }
      // Every tcgen05 operation issued above completes before this commit fires.
      commit(drain, 1);
      volatile int dummy = 0;
      dev::mbar_wait(drain, 0, &dummy, args.err);
    }
  } else if (warp >= kCopyWarp) {
    // ------------------------------------------------ scale-factor copiers (one thread each; the pair's leader)
    const int copier = warp - kCopyWarp;
    if (C::kBlockScaled && lane == 0 && leader) {
      // NVFP4: copier c takes the k-steps c, c + 2 (1 % faster than k-steps 2c, 2c + 1)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = !*abort_flag;
      int last = -1;
      uint32_t last_phase = 0;
      for (int tile = unit; tile < num_tiles && ok; tile += units) {
        for (int kt = 0; kt < args.k_tiles; ++kt) {
          // sf_full[stage] of this phase also means the MMAs that read the slot's previous
          // contents have completed (the producer refilled the stage only after they did)
          if (!dev::mbar_wait<kPair>(&sf_full[stage], phase, abort_flag, args.err)) {
            ok = false;
            break;
          }
          dev::tc_fence_after();
          issue_sf_copies(stage, copier, C::kSfCopiers);
          if (kPair) dev::tc_commit_pair(&sf_ready[stage], 1);
          else dev::tc_commit(&sf_ready[stage]);
          last = stage;
          last_phase = phase;
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
      }
      if (!ok && last >= 0) {
        // bounded wait for this thread's last copies before TMEM can be released
        volatile int dummy = 0;
        dev::mbar_wait<kPair>(&sf_ready[last], last_phase, &dummy, args.err);
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = smem + C::kSmemStage + (warp - 2) * 2048;
    const float alpha = (args.alpha_a ? __ldg(args.alpha_a) : 1.0f) * (args.alpha_b ? __ldg(args.alpha_b) : 1.0f);
    int it = 0;
    for (int tile = unit; tile < num_tiles; tile += units, ++it) {
      int mt, nt;
      tile_coords(tile, args.m_tiles, args.n_tiles, mt, nt, args.raster);
      const int as = it % C::kAccStages;
      const uint32_t aphase = static_cast<uint32_t>(it / C::kAccStages) & 1u;
      if (!dev::mbar_wait<kPair>(&acc_full[as], aphase, abort_flag, args.err)) break;
      dev::tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(as * BN + half * 128);
      uint32_t acc[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) dev::tmem_ld_32x32b_x32(taddr + 32 * c, acc[c]);
      dev::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) dev::reg_fence(acc[c]);
      // Release: every epilogue warp of both CTAs arrives on the leader's accumulator-empty
      // barrier as soon as its own loads are complete.  In a pair the arrival is a
      // tcgen05.commit multicast to the leader (it tracks no tcgen05 operation of this
      // thread: the loads above have completed); it reaches the leader's MMA thread about
      // 600 ns sooner than an mbarrier arrive at cluster scope, which matters for the
      // single-accumulator kinds (NVFP4 / MXFP8 5-11 % faster at K = 4096).
      dev::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        dev::tc_fence_after();
        if (kPair) dev::tc_commit_pair(&acc_empty[as], 1);
        else dev::mbar_arrive(&acc_empty[as]);
      }

      // Stage 32 rows x 64 bytes at a time in this warp's shared-memory box and write it
      // with a TMA store (the store clips rows >= M and columns >= N).
      const int m0 = (mt * CG + static_cast<int>(rank)) * BM + quarter * 32;
      const int n0 = nt * BN + half * 128;
      // One 32-row x 64-byte box: lane-row words w[0..15] -> staging buffer -> TMA store.
      auto store_box = [&](const uint32_t (&w)[16], int nb) {
        if (lane == 0) dev::bulk_wait_read0();  // the previous box has left the staging buffer
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = (j + (lane >> 1)) & 3;  // rotate chunk order: conflict-free 16-byte stores
          uint32_t v0 = w[0], v1 = w[1], v2 = w[2], v3 = w[3];
#pragma unroll
          for (int q = 1; q < 4; ++q)
            if (ch == q) v0 = w[4 * q], v1 = w[4 * q + 1], v2 = w[4 * q + 2], v3 = w[4 * q + 3];
          *reinterpret_cast<uint4*>(stg + lane * 64 + ch * 16) = make_uint4(v0, v1, v2, v3);
        }
        dev::fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          if (args.accumulate) dev::tma_reduce_add_2d(&tmD, stg, nb, m0);
          else dev::tma_store_2d(&tmD, stg, nb * (args.out_f32 ? 4 : 2), m0);
          dev::bulk_commit();
        }
      };
      if (m0 < args.M) {
        if (args.out_f32) {
#pragma unroll
          for (int bx = 0; bx < 8; ++bx) {
            const int nb = n0 + bx * 16;
            if (nb >= args.N) break;
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float b = args.bias ? __ldg(args.bias + nb + i) : 0.0f;
              w[i] = __float_as_uint(__fmaf_rn(__uint_as_float(acc[bx >> 1][(bx & 1) * 16 + i]), alpha, b));
            }
            store_box(w, nb);
          }
        } else {
#pragma unroll
          for (int bx = 0; bx < 4; ++bx) {
            const int nb = n0 + bx * 32;
            if (nb >= args.N) break;
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              // N is a multiple of 16: the box's second half may lie past N (the store
              // clips it), where the bias is not read
              const bool bin = args.bias && nb + 2 * i < args.N;
              const float b0 = bin ? __ldg(args.bias + nb + 2 * i) : 0.0f;
              const float b1 = bin ? __ldg(args.bias + nb + 2 * i + 1) : 0.0f;
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__fmaf_rn(__uint_as_float(acc[bx][2 * i]), alpha, b0),
                                                              __fmaf_rn(__uint_as_float(acc[bx][2 * i + 1]), alpha, b1));
              w[i] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            store_box(w, nb);
          }
        }
      }
    }
    if (lane == 0) dev::bulk_wait0();
  }

  dev::tc_fence_before();
  __syncthreads();
  if (kPair) dev::cluster_sync();  // the leader's MMAs read the peer's shared memory until here
  dev::tc_fence_after();
  if (warp == 1) {
    if (kPair) dev::tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else dev::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---- host launch ----------------------------------------------------------------------------------

// Instruction descriptor (tcgen05, dense): D format in bits 4-5 (F32 = 1) for the
// non-block-scaled kinds, A / B formats in bits 7-9 / 10-12, K-major operands
// (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28; for the
// block-scaled kinds bit 23 selects the scale format (UE8M0 = 1, UE4M3 = 0).
uint32_t make_idesc(int kind, uint32_t afmt, uint32_t bfmt, int m) {
  uint32_t d = 0;
  if (kind == kBF16 || kind == kFP8) d |= 1u << 4;
  d |= (afmt & 7u) << 7;
  d |= (bfmt & 7u) << 10;
  d |= static_cast<uint32_t>(BN >> 3) << 17;
  if (kind == kMXFP8) d |= 1u << 23;
  d |= static_cast<uint32_t>(m >> 4) << 24;
  return d;
}

template <int KIND, int CG = 1>
te_status launch_gemm(const void* A, const void* B, int64_t row_bytes, const uint8_t* sfa, const uint8_t* sfb,
                      int64_t sf_katoms, const float* alpha_a, const float* alpha_b, const float* bias, void* D,
                      te_dtype out, int accumulate, int64_t M, int64_t N, int64_t K, uint32_t afmt, uint32_t bfmt,
                      cudaStream_t st, int a_mn = 0, int b_mn = 0) {
  using C = Cfg<KIND, CG>;
  static bool attr_set[64] = {false};
  static int max_clusters[64] = {0};
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  if (dev_id < 0 || dev_id >= 64) return TE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemTotal;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!attr_set[dev_id]) {
    if (cudaFuncSetAttribute(gemm_kernel<KIND, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemTotal) !=
        cudaSuccess)
      return record_cuda(cudaGetLastError());
    int n = num_sms() / CG;
    if (CG > 1) {
      // clusters that can be resident at once (a GPC may leave an SM unpaired)
      cfg.gridDim = dim3(CG * n, 1, 1);
      int mc = 0;
      if (cudaOccupancyMaxActiveClusters(&mc, gemm_kernel<KIND, CG>, &cfg) != cudaSuccess || mc <= 0)
        return record_cuda(cudaGetLastError());
      n = mc < n ? mc : n;
    }
    max_clusters[dev_id] = n;
    attr_set[dev_id] = true;
  }
  CUtensorMap ta, tb;
  te_status s = a_mn ? make_tmap_2d(&ta, A, static_cast<uint64_t>(M) * 2, static_cast<uint64_t>(K), 64)
                     : make_tmap_2d(&ta, A, static_cast<uint64_t>(row_bytes), static_cast<uint64_t>(M), BM);
  if (s != TE_OK) return s;
  s = b_mn ? make_tmap_2d(&tb, B, static_cast<uint64_t>(N) * 2, static_cast<uint64_t>(K), 64)
           : make_tmap_2d(&tb, B, static_cast<uint64_t>(row_bytes), static_cast<uint64_t>(N), C::kBRows);
  if (s != TE_OK) return s;
  CUtensorMap td;
  const uint32_t esize = out == TE_F32 ? 4u : 2u;
  // accumulate: an fp32-typed map (the reduce-add needs the element type), box 16 x 32
  s = accumulate ? make_tmap_2d_f32(&td, static_cast<const float*>(D), static_cast<uint64_t>(N),
                                    static_cast<uint64_t>(M), 16u, 32u)
                 : make_tmap_2d_plain(&td, D, static_cast<uint64_t>(N) * esize, static_cast<uint64_t>(M), 64u, 32u);
  if (s != TE_OK) return s;
  // scale tensors as 256-byte rows (CTA pairs load them by TMA); unused otherwise
  CUtensorMap tsa = td, tsb = td;
  if (C::kBlockScaled && C::kPair) {
    const uint64_t rows_a = static_cast<uint64_t>((M + 127) / 128) * static_cast<uint64_t>(sf_katoms) * 2;
    const uint64_t rows_b = static_cast<uint64_t>((N + 127) / 128) * static_cast<uint64_t>(sf_katoms) * 2;
    if (rows_a >= (uint64_t(1) << 31) || rows_b >= (uint64_t(1) << 31)) return TE_ERR_SHAPE;
    s = make_tmap_2d_plain(&tsa, sfa, 256u, rows_a, 256u, static_cast<uint32_t>(2 * C::kSfAtoms));
    if (s != TE_OK) return s;
    s = make_tmap_2d_plain(&tsb, sfb, 256u, rows_b, 256u, static_cast<uint32_t>(2 * C::kSfAtoms));
    if (s != TE_OK) return s;
  }
  int* err = device_error_word();
  if (err == nullptr) return record_cuda(cudaErrorInvalidDevice);
  GemmArgs g;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.k_tiles = static_cast<int>((row_bytes + 127) / 128);
  g.m_tiles = static_cast<int>((M + BM * CG - 1) / (BM * CG));
  g.n_tiles = static_cast<int>((N + BN - 1) / BN);
  g.sfa = sfa;
  g.sfb = sfb;
  g.sf_katoms = sf_katoms;
  g.sfb_row_atoms = static_cast<int>((N + 127) / 128);
  g.alpha_a = alpha_a;
  g.alpha_b = alpha_b;
  g.bias = bias;
  g.D = D;
  g.out_f32 = out == TE_F32;
  g.accumulate = accumulate;
  g.idesc = make_idesc(KIND, afmt, bfmt, BM * CG) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16);
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  g.raster = (KIND != kBF16 && g.k_tiles >= 64 && g.m_tiles != g.n_tiles) ? 1 : 0;   // >= 8 KB of K per row
  g.err = err;
  const int tiles = g.m_tiles * g.n_tiles;
  // The fewest CTA pairs that keep the number of waves: every pair runs the same number of
  // tiles (within one), and the SMs left idle leave their share of the power budget to the
  // busy ones (FP8 / MXFP8 layer GEMMs 1.4-1.7 % faster than with one pair per two SMs).
  int units = tiles < max_clusters[dev_id] ? tiles : max_clusters[dev_id];
  if (units > 0) {
    const int waves = (tiles + units - 1) / units;
    units = (tiles + waves - 1) / waves;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(CG * units), 1, 1);
  if (cudaLaunchKernelEx(&cfg, gemm_kernel<KIND, CG>, ta, tb, td, tsa, tsb, g) != cudaSuccess)
    return record_cuda(cudaGetLastError());
  count_launch();
  return launch_status();
}

te_status check_gemm(const void* A, const void* B, const void* D, te_dtype out, int accumulate, int64_t M, int64_t N,
                     int64_t K, int64_t k_multiple) {
  if (out != TE_BF16 && out != TE_F32) return TE_ERR_DTYPE;
  if (accumulate != 0 && accumulate != 1) return TE_ERR_ARG;
  if (accumulate && out != TE_F32) return TE_ERR_DTYPE;
  if (M < 0 || N < 0 || K <= 0 || M % 16 || N % 16 || K % k_multiple) return TE_ERR_SHAPE;
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return TE_ERR_SHAPE;
  if (M * N == 0) return TE_OK;
  if (!A || !B || !D) return TE_ERR_NULL;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return TE_ERR_ALIGN;
  return TE_OK;
}

inline bool fp8_fmt(te_dtype f) { return f == TE_E4M3 || f == TE_E5M2; }
inline uint32_t f8_code(te_dtype f) { return f == TE_E5M2 ? 1u : 0u; }

}  // namespace
}  // namespace te

using namespace te;

extern "C" {

te_status te_gemm_bf16(const void* A, te_layout a_layout, const void* B, te_layout b_layout, const float* bias, void* D,
                       te_dtype out_dtype, int accumulate, int64_t M, int64_t N, int64_t K, void* stream) {
  if ((a_layout != TE_K_MAJOR && a_layout != TE_MN_MAJOR) || (b_layout != TE_K_MAJOR && b_layout != TE_MN_MAJOR))
    return TE_ERR_ARG;
  te_status s = check_gemm(A, B, D, out_dtype, accumulate, M, N, K, 16);
  if (s != TE_OK || M * N == 0) return s;
  return launch_gemm<kBF16, 2>(A, B, K * 2, nullptr, nullptr, 0, nullptr, nullptr, bias, D, out_dtype, accumulate, M, N,
                               K, 1u, 1u, static_cast<cudaStream_t>(stream), a_layout == TE_MN_MAJOR,
                               b_layout == TE_MN_MAJOR);
}

te_status te_gemm_fp8(const uint8_t* A, te_dtype fa, const uint8_t* B, te_dtype fb, const float* a_scale_inv,
                      const float* b_scale_inv, const float* bias, void* D, te_dtype out_dtype, int accumulate,
                      int64_t M, int64_t N, int64_t K, void* stream) {
  if (!fp8_fmt(fa) || !fp8_fmt(fb)) return TE_ERR_DTYPE;
  te_status s = check_gemm(A, B, D, out_dtype, accumulate, M, N, K, 16);
  if (s != TE_OK || M * N == 0) return s;
  if (!a_scale_inv || !b_scale_inv) return TE_ERR_NULL;
  return launch_gemm<kFP8, 2>(A, B, K, nullptr, nullptr, 0, a_scale_inv, b_scale_inv, bias, D, out_dtype, accumulate, M,
                              N, K, f8_code(fa), f8_code(fb), static_cast<cudaStream_t>(stream));
}

te_status te_gemm_mxfp8(const uint8_t* A, te_dtype fa, const uint8_t* sA, const uint8_t* B, te_dtype fb,
                        const uint8_t* sB, const float* bias, void* D, te_dtype out_dtype, int accumulate,
                        int64_t M, int64_t N, int64_t K, void* stream) {
  if (!fp8_fmt(fa) || !fp8_fmt(fb)) return TE_ERR_DTYPE;
  te_status s = check_gemm(A, B, D, out_dtype, accumulate, M, N, K, 32);
  if (s != TE_OK || M * N == 0) return s;
  if (!sA || !sB) return TE_ERR_NULL;
  if (!aligned16(sA) || !aligned16(sB)) return TE_ERR_ALIGN;
  const int64_t katoms = ((K / 32 + 3) / 4);
  return launch_gemm<kMXFP8, 2>(A, B, K, sA, sB, katoms, nullptr, nullptr, bias, D, out_dtype, accumulate, M, N, K,
                                f8_code(fa), f8_code(fb), static_cast<cudaStream_t>(stream));
}

te_status te_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const float* gA, const uint8_t* B, const uint8_t* sB,
                        const float* gB, const float* bias, void* D, te_dtype out_dtype, int accumulate,
                        int64_t M, int64_t N, int64_t K, void* stream) {
  te_status s = check_gemm(A, B, D, out_dtype, accumulate, M, N, K, 32);
  if (s != TE_OK || M * N == 0) return s;
  if (!sA || !sB || !gA || !gB) return TE_ERR_NULL;
  if (!aligned16(sA) || !aligned16(sB)) return TE_ERR_ALIGN;
  const int64_t katoms = ((K / 16 + 15) / 16) * 4;
  return launch_gemm<kNVFP4, 2>(A, B, K / 2, sA, sB, katoms, gA, gB, bias, D, out_dtype, accumulate, M, N, K, 1u, 1u,
                                static_cast<cudaStream_t>(stream));
}

}  // extern "C"
