// weights.cu -- the layer weights handle: canonical NVFP4 expert matrices
// repacked once into the layouts the kernels read.
//
// Each expert is an independent FFN with its own gate, up and down matrices
// (page "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算", MoE core
// mechanism), stored as NVFP4 (page "8GB 笔记本 39.3 tok/s、单卡跑 753B：
// FreeToken 把 frontier MoE 拉回本地", sections 实测六款消费级硬件 and 局限).
// The canonical form a caller holds is one row-major matrix per projection:
// codes [N][K/2] (element 2j in the low nibble of byte j), E4M3 scales
// [N][K/16] and an fp32 tensor scale.  The handle owns device copies in the
// requested kernel layouts:
//   FT_LAYOUT_ROWS          gate and up interleaved row by row ([2I][H]), down as is;
//   FT_LAYOUT_DECODE_TILES  the same matrices in 16-row tiles (ft_nvfp4_pack_tiles);
//   FT_LAYOUT_UMMA_TILES    the same matrices in 128x128 blocks (ft_nvfp4_pack_umma);
// plus one array of tensor scales {gate, up, down, 0} per expert shared by all
// layouts.  Repacking is a byte permutation: the kernels compute on exactly the
// caller's codes and scales.
#include "common.cuh"

#include <new>

struct ft_moe_weights {
    int E, H, I, flags;
    uint8_t* gu[3];       // per layout: gate/up bytes of all experts (nullptr if not requested)
    uint8_t* dn[3];       // per layout: down bytes
    uint8_t* gu_sc;       // ROWS layout: gate/up scales [E][2I][H/16]
    uint8_t* dn_sc;       // ROWS layout: down scales [E][H][I/16]
    int64_t gu_stride, dn_stride, gu_sc_stride, dn_sc_stride;
    float* tscale;        // [E][4]
};

namespace ft {

static bool check_matrix(const ft_nvfp4_matrix& m, int64_t N, int64_t K) {
    (void)N;
    return m.codes && m.scales && m.tensor_scale && aligned(m.codes, 16) && m.codes_ld % 16 == 0 &&
           m.codes_ld >= K / 2 && m.scales_ld >= K / 16 && aligned(m.tensor_scale, 4);
}

static void free_weights(ft_moe_weights* w) {
    if (!w) return;
    for (int l = 0; l < 3; ++l) {
        if (w->gu[l]) cudaFree(w->gu[l]);
        if (w->dn[l]) cudaFree(w->dn[l]);
    }
    if (w->gu_sc) cudaFree(w->gu_sc);
    if (w->dn_sc) cudaFree(w->dn_sc);
    if (w->tscale) cudaFree(w->tscale);
    delete w;
}

}  // namespace ft

using namespace ft;

extern "C" {

ft_status ft_moe_weights_create(const ft_nvfp4_expert_desc* experts, int E, int H, int I, int layout_flags,
                                ft_stream_t stream, ft_moe_weights** out) {
    const char* fn = "ft_moe_weights_create";
    if (!out) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": out is null");
    *out = nullptr;
    if (!experts) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": experts is null");
    if (E <= 0 || E > 1024 || H <= 0 || H % 256 || I <= 0 || I % 128)
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": need 1 <= E <= 1024, H a multiple of 256, I a multiple of 128");
    const int all = FT_WEIGHTS_ROWS | FT_WEIGHTS_DECODE_TILES | FT_WEIGHTS_UMMA_TILES;
    if (layout_flags == 0 || (layout_flags & ~all))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": layout_flags must be a non-empty set of FT_WEIGHTS_*");
    for (int e = 0; e < E; ++e)
        if (!check_matrix(experts[e].gate, I, H) || !check_matrix(experts[e].up, I, H) ||
            !check_matrix(experts[e].down, H, I))
            return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": expert " + std::to_string(e) +
                                                ": null pointer, codes not 16-byte aligned, or a row stride too small");
    ft_moe_weights* w = new (std::nothrow) ft_moe_weights();
    if (!w) return fail(FT_ERR_OOM, std::string(fn) + ": host allocation failed");
    w->E = E;
    w->H = H;
    w->I = I;
    w->flags = layout_flags;
    const int64_t gu_bytes = (int64_t)2 * I * H * 9 / 16, dn_bytes = (int64_t)H * I * 9 / 16;
    w->gu_stride = (gu_bytes + 255) / 256 * 256;
    w->dn_stride = (dn_bytes + 255) / 256 * 256;
    w->gu_sc_stride = ((int64_t)2 * I * (H / 16) + 255) / 256 * 256;
    w->dn_sc_stride = ((int64_t)H * (I / 16) + 255) / 256 * 256;
    // the ROWS layout is the source of the tiled ones; without ROWS, one expert's worth is staged
    const bool keep_rows = layout_flags & FT_WEIGHTS_ROWS;
    const int64_t row_codes_gu = (int64_t)2 * I * (H / 2), row_codes_dn = (int64_t)H * (I / 2);
    const int64_t nrows = keep_rows ? E : 1;
    cudaError_t err = cudaSuccess;
    auto take = [&](void** p, size_t bytes) {
        if (err == cudaSuccess) err = cudaMalloc(p, bytes);
    };
    take((void**)&w->gu[FT_LAYOUT_ROWS], (size_t)(nrows * ((row_codes_gu + 255) / 256 * 256)));
    take((void**)&w->dn[FT_LAYOUT_ROWS], (size_t)(nrows * ((row_codes_dn + 255) / 256 * 256)));
    take((void**)&w->gu_sc, (size_t)(nrows * w->gu_sc_stride));
    take((void**)&w->dn_sc, (size_t)(nrows * w->dn_sc_stride));
    if (layout_flags & FT_WEIGHTS_DECODE_TILES) {
        take((void**)&w->gu[FT_LAYOUT_DECODE_TILES], (size_t)(E * w->gu_stride));
        take((void**)&w->dn[FT_LAYOUT_DECODE_TILES], (size_t)(E * w->dn_stride));
    }
    if (layout_flags & FT_WEIGHTS_UMMA_TILES) {
        take((void**)&w->gu[FT_LAYOUT_UMMA_TILES], (size_t)(E * w->gu_stride));
        take((void**)&w->dn[FT_LAYOUT_UMMA_TILES], (size_t)(E * w->dn_stride));
    }
    take((void**)&w->tscale, (size_t)E * 4 * sizeof(float));
    if (err != cudaSuccess) {
        cudaGetLastError();
        free_weights(w);
        return fail(FT_ERR_OOM, std::string(fn) + ": device allocation failed: " + cudaGetErrorString(err));
    }
    const int64_t rc_gu = (row_codes_gu + 255) / 256 * 256, rc_dn = (row_codes_dn + 255) / 256 * 256;
    cudaStream_t s = cu(stream);
    ft_status st = FT_OK;
    err = cudaMemsetAsync(w->tscale, 0, (size_t)E * 4 * sizeof(float), s);
    for (int e = 0; e < E && err == cudaSuccess && st == FT_OK; ++e) {
        const ft_nvfp4_expert_desc& x = experts[e];
        const int64_t r = keep_rows ? e : 0;
        uint8_t* guc = w->gu[FT_LAYOUT_ROWS] + r * rc_gu;
        uint8_t* gus = w->gu_sc + r * w->gu_sc_stride;
        uint8_t* dnc = w->dn[FT_LAYOUT_ROWS] + r * rc_dn;
        uint8_t* dns = w->dn_sc + r * w->dn_sc_stride;
        // gate row i -> row 2i, up row i -> row 2i+1 of the [2I][H] gate/up matrix
        const cudaMemcpyKind d2d = cudaMemcpyDeviceToDevice;
        if (err == cudaSuccess) err = cudaMemcpy2DAsync(guc, H, x.gate.codes, x.gate.codes_ld, H / 2, I, d2d, s);
        if (err == cudaSuccess) err = cudaMemcpy2DAsync(guc + H / 2, H, x.up.codes, x.up.codes_ld, H / 2, I, d2d, s);
        if (err == cudaSuccess) err = cudaMemcpy2DAsync(gus, H / 8, x.gate.scales, x.gate.scales_ld, H / 16, I, d2d, s);
        if (err == cudaSuccess) err = cudaMemcpy2DAsync(gus + H / 16, H / 8, x.up.scales, x.up.scales_ld, H / 16, I, d2d, s);
        if (err == cudaSuccess) err = cudaMemcpy2DAsync(dnc, I / 2, x.down.codes, x.down.codes_ld, I / 2, H, d2d, s);
        if (err == cudaSuccess) err = cudaMemcpy2DAsync(dns, I / 16, x.down.scales, x.down.scales_ld, I / 16, H, d2d, s);
        float* ts = w->tscale + (int64_t)e * 4;
        if (err == cudaSuccess) err = cudaMemcpyAsync(ts + 0, x.gate.tensor_scale, sizeof(float), d2d, s);
        if (err == cudaSuccess) err = cudaMemcpyAsync(ts + 1, x.up.tensor_scale, sizeof(float), d2d, s);
        if (err == cudaSuccess) err = cudaMemcpyAsync(ts + 2, x.down.tensor_scale, sizeof(float), d2d, s);
        if (err != cudaSuccess) break;
        if (layout_flags & FT_WEIGHTS_DECODE_TILES) {
            st = ft_nvfp4_pack_tiles(guc, H / 2, gus, H / 16, 2 * I, H, w->gu[FT_LAYOUT_DECODE_TILES] + e * w->gu_stride,
                                     stream);
            if (st == FT_OK)
                st = ft_nvfp4_pack_tiles(dnc, I / 2, dns, I / 16, H, I, w->dn[FT_LAYOUT_DECODE_TILES] + e * w->dn_stride,
                                         stream);
        }
        if (st == FT_OK && (layout_flags & FT_WEIGHTS_UMMA_TILES)) {
            st = ft_nvfp4_pack_umma(guc, H / 2, gus, H / 16, 2 * I, H, w->gu[FT_LAYOUT_UMMA_TILES] + e * w->gu_stride,
                                    stream);
            if (st == FT_OK)
                st = ft_nvfp4_pack_umma(dnc, I / 2, dns, I / 16, H, I, w->dn[FT_LAYOUT_UMMA_TILES] + e * w->dn_stride,
                                        stream);
        }
    }
    if (err == cudaSuccess && st == FT_OK) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess || st != FT_OK) {
        const std::string why = err != cudaSuccess ? std::string(cudaGetErrorString(err)) : std::string(ft_last_error());
        cudaGetLastError();
        cudaStreamSynchronize(s);
        free_weights(w);
        return fail(FT_ERR_CUDA, std::string(fn) + ": repacking failed: " + why);
    }
    if (!keep_rows) {  // the staging copy of one expert is no longer needed
        cudaFree(w->gu[FT_LAYOUT_ROWS]);
        cudaFree(w->dn[FT_LAYOUT_ROWS]);
        cudaFree(w->gu_sc);
        cudaFree(w->dn_sc);
        w->gu[FT_LAYOUT_ROWS] = w->dn[FT_LAYOUT_ROWS] = w->gu_sc = w->dn_sc = nullptr;
    }
    *out = w;
    return FT_OK;
}

ft_status ft_moe_weights_describe(const ft_moe_weights* w, int layout, ft_moe_layer_weights* desc) {
    const char* fn = "ft_moe_weights_describe";
    if (!w || !desc) return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": null pointer");
    if (layout < 0 || layout > 2 || !(w->flags & (1 << layout)))
        return fail(FT_ERR_INVALID_ARG, std::string(fn) + ": the handle holds no copy in that layout");
    *desc = ft_moe_layer_weights{};
    desc->E = w->E;
    desc->H = w->H;
    desc->I = w->I;
    desc->n_weights = w->E;
    desc->layout = layout;
    desc->gu_codes = w->gu[layout];
    desc->d_codes = w->dn[layout];
    if (layout == FT_LAYOUT_ROWS) {
        desc->gu_codes_stride = ((int64_t)2 * w->I * (w->H / 2) + 255) / 256 * 256;
        desc->d_codes_stride = ((int64_t)w->H * (w->I / 2) + 255) / 256 * 256;
        desc->gu_scales = w->gu_sc;
        desc->gu_scales_stride = w->gu_sc_stride;
        desc->d_scales = w->dn_sc;
        desc->d_scales_stride = w->dn_sc_stride;
    } else {
        desc->gu_codes_stride = w->gu_stride;
        desc->d_codes_stride = w->dn_stride;
    }
    desc->tscale = w->tscale;
    desc->tscale_stride = 4;
    return FT_OK;
}

ft_status ft_moe_weights_destroy(ft_moe_weights* w) {
    if (!w) return FT_OK;
    free_weights(w);
    return FT_OK;
}

}  // extern "C"
