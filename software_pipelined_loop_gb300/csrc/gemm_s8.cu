// gemm_s8.cu -- INT8 variants: fp16-widened operands, chunked exact int32 epilogue.
#include "launch_impl.cuh"

namespace gp {

static const Variant kS8Variants[] = {
    make_variant<GemmCfg<256, 4, false, true>>(),  // fp16-widened operands from the workspace
    make_variant<GemmCfg<256, 6, false, true, false, 1, true>>(),  // CTA pair, 256x256 tiles
    make_variant<GemmCfg<256, 6, false, true, false, 1, true, 1, 4, false, true>>(),  // quad: two pairs share A
    make_variant<GemmCfg<256, 3, false, true, false, 1, true, 1, 4, false, false, 128>>(),  // pair, 128 k per stage
    make_variant<GemmCfg<128, 6, false, true>>(),
    make_variant<GemmCfg<256, 2, false, true, true, 4>>(),  // int8 TMA + in-kernel widening
    make_variant<GemmCfg<128, 3, false, true, true, 6>>(),
    make_variant<GemmCfg<256, 4, false, true, true, 4, true, 1, 2>>(),  // CTA pair + in-kernel widening (opt-in)
};

int variants_s8(const Variant **out)
{
    *out = kS8Variants;
    return static_cast<int>(sizeof(kS8Variants) / sizeof(kS8Variants[0]));
}

}  // namespace gp
