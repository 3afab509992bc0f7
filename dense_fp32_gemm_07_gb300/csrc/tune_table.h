// tune_table.h -- shape-keyed plan choice, frozen from measurements on GB300.
//
// The handbook (section 接下来的优化方向, 参数自动调优) notes that the best block
// and thread tile sizes depend on the GPU and on the matrix shape and that real
// libraries keep a configuration per shape; this table is that configuration.
// Rules are tried in order; the first whose class and bounds match names the
// plan.  "fast" = both operands bulk-tensor eligible (16-byte aligned, lda, ldb
// and K multiples of 4, no op() on B); "general" = anything else.
#pragma once

namespace b2g {

enum OperandClass : int { kClassFast = 0, kClassFastTransA = 1, kClassGeneral = 2 };

struct TuneRule {
  int cls;
  int m_min, m_max;  // inclusive bounds on M
  int n_min, n_max;  // inclusive bounds on N
  const char* plan;
};

constexpr int kInf = 0x7fffffff;

// Measured on GB300 (152 SMs); see the bench sweep notes in the design document.
const TuneRule kTuneTable[] = {
    {kClassFast, 0, 48, 0, kInf, "tma_32x64x32_s6"},
    {kClassFast, 49, 127, 0, kInf, "tma_64x128x16_s6"},
    {kClassFast, 128, kInf, 0, 127, "tma_64x128x16_s6"},
    {kClassFast, 128, kInf, 128, kInf, "tma_128x128x16_s6"},
    {kClassFastTransA, 0, kInf, 0, kInf, "tmaT_128x128x16_s6"},
    {kClassGeneral, 0, 96, 0, kInf, "gen_64x64x16_s4"},
    {kClassGeneral, 97, kInf, 0, 96, "gen_64x64x16_s4"},
    {kClassGeneral, 97, kInf, 97, kInf, "gen_128x128x16_s4"},
};

}  // namespace b2g
