// prompt.cu -- placeholder, replaced by the tcgen05 prompt kernel.
#include "common.cuh"
extern "C" int attn_prompt_q8(const uint16_t*, int, int, const kvq8_cache*, int, int, float, float*, kvq8_stream_t) {
    return KVQ8_ERR_UNSUPPORTED;
}
