// The instantiations of gqa_simt_f32_small.cu in their plain single-token form
// (no multi-token step, no window), compiled without the multi-token schedule
// branches.
#define GQA_MULTI_TOKEN 0
#define GQA_SIMT_GEN 0
#include "gqa_simt_f32_small.cu"
