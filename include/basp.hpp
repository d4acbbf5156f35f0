// basp.hpp -- header-only C++ convenience layer over the C ABI in basp.h.
//
// Adds nothing to what the C entry points do: basp::Layout owns a handle
// (destroyed with the object), exposes its basp_info, and forwards to the C
// calls, turning a non-OK status into a basp::Error that carries the status
// code.  All arguments, layouts and rules are those of basp.h.
#ifndef BASP_HPP
#define BASP_HPP

#include <stdexcept>
#include <string>
#include <utility>

#include "basp.h"

namespace basp {

class Error : public std::runtime_error {
public:
    Error(basp_status status, const char *where)
        : std::runtime_error(std::string(where) + ": " + basp_status_string(status)),
          status_(status) {}
    basp_status status() const { return status_; }

private:
    basp_status status_;
};

inline void check(basp_status s, const char *where) {
    if (s != BASP_OK) throw Error(s, where);
}

class Layout {
public:
    // K = 0 asks for the BASP rule K = N / B.
    Layout(int64_t B, int64_t S, int64_t Hq, int64_t Hkv, int64_t d, int64_t N,
           int64_t K, basp_dtype dtype = BASP_DTYPE_BF16,
           basp_order order = BASP_ORDER_BSHD) {
        const basp_layout_desc desc = {B, S, Hq, Hkv, d, N, K, dtype, order};
        check(basp_layout_create_ex(&desc, &handle_), "basp_layout_create_ex");
        check(basp_layout_query(handle_, &info_), "basp_layout_query");
    }
    ~Layout() { basp_layout_destroy(handle_); }
    Layout(const Layout &) = delete;
    Layout &operator=(const Layout &) = delete;
    Layout(Layout &&o) noexcept : handle_(o.handle_), info_(o.info_) { o.handle_ = nullptr; }
    Layout &operator=(Layout &&o) noexcept {
        std::swap(handle_, o.handle_);
        std::swap(info_, o.info_);
        return *this;
    }

    const basp_layout *handle() const { return handle_; }
    const basp_info &info() const { return info_; }

    // seq-sharded -> head-sharded (any of the three pairs may be null)
    void seq2head(const void *q, const void *k, const void *v, void *q_out,
                  void *k_out, void *v_out, cudaStream_t stream,
                  basp_algo algo = BASP_ALGO_FUSED, void *workspace = nullptr,
                  size_t workspace_bytes = 0) const {
        check(basp_seq2head(handle_, algo, q, k, v, q_out, k_out, v_out, workspace,
                            workspace_bytes, stream), "basp_seq2head");
    }
    // head-sharded -> seq-sharded
    void head2seq(const void *o, const void *k, const void *v, void *o_out,
                  void *k_out, void *v_out, cudaStream_t stream,
                  basp_algo algo = BASP_ALGO_FUSED, void *workspace = nullptr,
                  size_t workspace_bytes = 0) const {
        check(basp_head2seq(handle_, algo, o, k, v, o_out, k_out, v_out, workspace,
                            workspace_bytes, stream), "basp_head2seq");
    }
    // packed QKV projection output -> head-sharded Q, K, V, and back
    void seq2head_qkv(const void *qkv, void *q_out, void *k_out, void *v_out,
                      cudaStream_t stream) const {
        check(basp_seq2head_qkv(handle_, qkv, q_out, k_out, v_out, stream),
              "basp_seq2head_qkv");
    }
    void head2seq_qkv(const void *q, const void *k, const void *v, void *qkv_out,
                      cudaStream_t stream) const {
        check(basp_head2seq_qkv(handle_, q, k, v, qkv_out, stream), "basp_head2seq_qkv");
    }
    // host buffers in and out: staged through caller-owned device `staging`,
    // or (staging null) read and written in place when page-locked
    void seq2head_host(const void *q, const void *k, const void *v, void *q_out,
                       void *k_out, void *v_out, void *staging, size_t staging_bytes,
                       cudaStream_t stream, basp_algo algo = BASP_ALGO_FUSED,
                       void *workspace = nullptr, size_t workspace_bytes = 0) const {
        check(basp_seq2head_host(handle_, algo, q, k, v, q_out, k_out, v_out, staging,
                                 staging_bytes, workspace, workspace_bytes, stream),
              "basp_seq2head_host");
    }
    void head2seq_host(const void *o, const void *k, const void *v, void *o_out,
                       void *k_out, void *v_out, void *staging, size_t staging_bytes,
                       cudaStream_t stream, basp_algo algo = BASP_ALGO_FUSED,
                       void *workspace = nullptr, size_t workspace_bytes = 0) const {
        check(basp_head2seq_host(handle_, algo, o, k, v, o_out, k_out, v_out, staging,
                                 staging_bytes, workspace, workspace_bytes, stream),
              "basp_head2seq_host");
    }

private:
    basp_layout *handle_ = nullptr;
    basp_info info_{};
};

}  // namespace basp

#endif  // BASP_HPP
