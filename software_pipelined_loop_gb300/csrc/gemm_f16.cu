// gemm_f16.cu -- fp16 x fp16 -> fp32 variants of the pipelined GEMM.
#include "launch_impl.cuh"

namespace gp {

static const Variant kF16Variants[] = {
    make_variant<GemmCfg<256, 4, false, false>>(),  // TMA producer, 128x256 tiles
    make_variant<GemmCfg<256, 6, false, false, false, 1, true>>(),  // CTA pair, 256x256 tiles
    // CTA pair, 256x256 tiles, 128 k per stage (three 64 KiB stages).
    make_variant<GemmCfg<256, 3, false, false, false, 1, true, 1, 4, false, false, 128>>(),
    // Quad: two CTA pairs (256x512 tile) sharing A by multicast.
    make_variant<GemmCfg<256, 6, false, false, false, 1, true, 1, 4, false, true>>(),
    // CTA pair, 256x512 tiles: two N = 256 MMAs per k-step into one
    // 512-column accumulator; 48 B of operands per MMA cycle per SM instead
    // of 64, under what an SM can take in.
    make_variant<GemmCfg<512, 4, false, false, false, 1, true>>(),
    // Ring-depth ablation: 1 = load, wait, compute (no overlap); 2 = the
    // classic double buffer; 3 to 5.
    make_variant<GemmCfg<256, 1, false, false, false, 1, true>>(),
    make_variant<GemmCfg<256, 2, false, false, false, 1, true>>(),
    make_variant<GemmCfg<256, 3, false, false, false, 1, true>>(),
    make_variant<GemmCfg<256, 4, false, false, false, 1, true>>(),
    make_variant<GemmCfg<256, 5, false, false, false, 1, true>>(),
    make_variant<GemmCfg<128, 6, false, false>>(),  // TMA producer, 128x128 tiles (N <= 128)
    // The same tiles with 128 k per stage (three 64 KiB stages): each A row
    // is read 256 bytes at a time (plan override bk = 128).
    make_variant<GemmCfg<128, 3, false, false, false, 1, false, 1, 4, false, false, 128>>(),
    make_variant<GemmCfg<256, 4, true, false>>(),   // bounded-load producer (misaligned inputs)
    make_variant<GemmCfg<128, 6, true, false>>(),
    // Copies of the pair kernels at 6 and 1 stages that stamp the
    // pipelining trace (taken only while the trace hook is armed).
    make_variant<GemmCfg<256, 6, false, false, false, 1, true, 1, 4, true>>(),
    make_variant<GemmCfg<256, 1, false, false, false, 1, true, 1, 4, true>>(),
    make_variant<GemmCfg<512, 4, false, false, false, 1, true, 1, 4, true>>(),
    make_variant<GemmCfg<256, 6, false, false, false, 1, true, 1, 4, true, true>>(),
};

int variants_f16(const Variant **out)
{
    *out = kF16Variants;
    return static_cast<int>(sizeof(kF16Variants) / sizeof(kF16Variants[0]));
}

}  // namespace gp
