// tune_table.h -- shape-keyed plan choice, frozen from measurements on GB300.
//
// The handbook (section 接下来的优化方向, 参数自动调优) notes that the best block
// and thread tile sizes depend on the GPU and on the matrix shape and that real
// libraries keep a configuration per shape; this table is that configuration.
// Rules are tried in order; the first whose class and bounds match names the
// plan (for a strided batch whose products have at least 5e7 multiply-adds
// each, M*N*K counts the whole call: times the batch count).  "fast" = both
// operands bulk-tensor eligible (16-byte aligned, lda, ldb and K multiples of
// 4, no op() on B); "fast, B transposed" = the same alignment with op(B) = B^T;
// "general" = anything else.
#pragma once

namespace b2g {

enum OperandClass : int {
  kClassFast = 0,        // row-major A and B, bulk-tensor eligible
  kClassFastTransA = 1,  // A stored K x M, B row-major, bulk-tensor eligible
  kClassGeneral = 2,     // anything else
  kClassFastTransB = 3,  // B stored N x K (A either way), 16-byte aligned, lda, ldb, K % 4 == 0
};

struct TuneRule {
  int cls;
  int m_min, m_max;  // inclusive bounds on M
  int n_min, n_max;  // inclusive bounds on N
  double mnk_min;    // smallest M*N*K the rule applies to
  const char* plan;
  const char* fallback;  // plan used when `plan` needs a workspace that cannot be had
  double mnk_max = 1e300;  // the rule applies while M*N*K < mnk_max
};

constexpr int kInf = 0x7fffffff;

// Chosen from per-plan timings on GB300 (152 SMs) over the square sweep
// (128^3 .. 8192^3), the 8192x11008x4096 and 16x4096x4096 shapes and the
// ragged 1000x1025x777 shape.
const TuneRule kTuneTable[] = {
    // skinny M (N % 4 == 0): split-K.  From N = 2048 (16 column slabs) the
    // bulk-tensor fed plans whose k slabs add up inside a cluster of <= 8
    // CTAs; below, B streamed from global memory with up to one resident wave
    // of k splits and a reduction kernel (more k parallelism than 8 slabs)
    {kClassFast, 0, 8, 2048, kInf, 0, "skinnyT_m8", nullptr},
    {kClassFast, 9, 16, 2048, kInf, 0, "skinnyT_m16", nullptr},
    {kClassFast, 17, 32, 2048, kInf, 0, "skinnyT_m32", nullptr},
    {kClassFast, 0, 8, 0, kInf, 0, "skinny_m8", nullptr},
    {kClassFast, 9, 16, 0, kInf, 0, "skinny_m16", nullptr},
    {kClassFast, 17, 32, 0, kInf, 0, "skinny_m32", nullptr},
    // up to ~1.5e9 multiply-adds: one launch, one CTA per small output tile
    // with its k range split between the CTA's warps (32 x 64, 64 x 64 or
    // 64 x 128 tiles, whichever a wave model expects faster), unless the
    // split-tail plan of a later rule is expected faster (few tiles over a
    // long k range, or many waves)
    {kClassFast, 0, kInf, 0, kInf, 0, "wk_32x64x32_g8", nullptr, 1.5e9},
    // the transpose costs about what it saves here; the packed-FMA form of
    // the k-chunked kernel (two CTAs per SM) beats the scalar one by 0.35-0.9
    // us a call (128^3 8.52 -> 7.71 us, 512^3 13.66 -> 13.31, 1000 x 1024 x
    // 776 43.5 -> 42.1; CUDA-graph replay)
    {kClassFast, 0, kInf, 0, kInf, 0, "tma_64x128x16_s6_o5", nullptr, 1.0e9},
    // larger: A transposed into the workspace, then the transposed-layout
    // kernel (its 64 x 128 twin when that pads less, e.g. M <= 64)
    {kClassFast, 0, kInf, 0, kInf, 1.0e9, "pre_128x64x32_s3_o5", "tmaX_128x128x16_s6_o2"},
    // op(A) = A^T: small products in one launch (the wk kernel reading A
    // stored K x M), larger ones on the transposed-layout kernel
    {kClassFastTransA, 0, kInf, 0, kInf, 0, "wkT_32x64x32_g8", nullptr, 1.5e9},
    {kClassFastTransA, 0, kInf, 0, kInf, 0, "tmaT_128x64x32_s3_o5", nullptr},
    // op(B) = B^T on aligned operands: B^T (and A, unless it comes stored
    // K x M) transposed into the workspace by the 16-byte-vector transpose,
    // then the wk kernel (one launch) or the transposed-layout kernel
    // (4096^3: packing both operands with 4-byte moves cost 3.5% of the
    // call); small calls take the 4-byte feed
    {kClassFastTransB, 0, kInf, 0, kInf, 5.0e7, "wkR_32x64x32_g8", "gen_64x64x16_s4", 1.5e9},
    {kClassFastTransB, 0, kInf, 0, kInf, 5.0e7, "pret_128x64x32_s3_o5", "gen_64x64x16_s4"},
    // below 5e7 multiply-adds one packing launch for both operands beats the
    // two transposes, and either beats the 4-byte feed 2-4x (128^3 6.9 / 8.5 /
    // 14.6 us, 300^3 8.3 / 9.2 / 19.0), which stays the fallback without a
    // workspace
    {kClassFastTransB, 0, kInf, 0, kInf, 0, "wkP_32x64x32_g8", "gen_64x64x16_s4", 5.0e7},
    {kClassFastTransB, 0, kInf, 0, kInf, 0, "gen_64x64x16_s4", nullptr},
    // anything else (misaligned pointers, odd leading dimensions, K % 4 != 0,
    // op(B) = B^T): pack A^T and B aligned into the workspace, then the wk
    // kernel (one launch) or the transposed-layout kernel; the 4-byte feed
    // needs no workspace and is the fallback (128 x 128 x 127: packed + wk
    // 7.5 us, 4-byte feed 33.2; 300 x 300 x 301: 9.8 against 19.5)
    {kClassGeneral, 0, kInf, 0, kInf, 0, "wkP_32x64x32_g8", "gen_64x64x16_s4", 1.5e9},
    {kClassGeneral, 0, kInf, 0, kInf, 5.0e7, "pack_128x64x32_s3_o5", "gen_64x64x16_s4"},
    {kClassGeneral, 0, kInf, 0, kInf, 0, "gen_64x64x16_s4", nullptr},
};

}  // namespace b2g
