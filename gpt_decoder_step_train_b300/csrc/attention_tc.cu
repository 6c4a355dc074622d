// attention_tc.cu -- placeholder until the tensor-core attention lands.
#include "common.cuh"
namespace gpt2k {
bool attention_tc_supported(int) { return false; }
int attention_tc_forward(float*, float*, const float*, int, int, int, int, int*, cudaStream_t) { return GPT2_ENOTSUP; }
int attention_tc_backward(float*, const float*, const float*, const float*, const float*, int, int, int, int, int*, cudaStream_t) { return GPT2_ENOTSUP; }
}  // namespace gpt2k
