// api.cu -- host-only entry points of libcpthd: status strings, the
// value-based pad_between_seqs detector, host metadata validation, the
// host-known valid end that gates the tail-zeroing, and the device status
// word query.
#include <algorithm>
#include <vector>

#include "common.cuh"

extern "C" const char* cp_status_string(int status) {
  switch (status) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG";
    case CP_ERR_DIVISIBILITY: return "CP_ERR_DIVISIBILITY";
    case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED";
    case CP_ERR_ALIGNMENT: return "CP_ERR_ALIGNMENT";
    case CP_ERR_CUDA: return "CP_ERR_CUDA";
    case CP_ERR_WORKSPACE: return "CP_ERR_WORKSPACE";
    case CP_ERR_METADATA: return "CP_ERR_METADATA";
    case CP_ERR_TIMEOUT: return "CP_ERR_TIMEOUT";
    case CP_ERR_RANGE: return "CP_ERR_RANGE";
    default: return "CP_ERR_UNKNOWN";
  }
}

extern "C" int cp_version(void) { return 200; }

// "THD P2P context-parallel regression when padded cu_seqlens are value-equal
// but not object-identical", §Expected behavior: equal values mean no padding
// between sequences, whatever the objects are.
extern "C" int cp_detect_pad_between_seqs(const int32_t* cu_host, const int32_t* cup_host,
                                          int n_docs, int* out) {
  if (!cu_host || !out || n_docs < 0) return CP_ERR_INVALID_ARG;
  int pad = 0;
  if (cup_host)
    for (int i = 0; i <= n_docs; ++i)
      if (cu_host[i] != cup_host[i]) { pad = 1; break; }
  *out = pad;
  return CP_OK;
}

extern "C" int cp_validate_seqlens(const int32_t* cu, const int32_t* cup, int n_docs,
                                   int64_t total_tokens, int cp_size, cp_strategy_t strategy,
                                   int pad) {
  if (!cup || (pad && !cu) || n_docs < 1 || cp_size < 1) return CP_ERR_INVALID_ARG;
  if (strategy != CP_DUAL_CHUNK_SWAP && strategy != CP_NO_LOAD_BALANCE) return CP_ERR_INVALID_ARG;
  if (cup[0] != 0 || cup[n_docs] != total_tokens) return CP_ERR_METADATA;
  if (pad && cu[0] != 0) return CP_ERR_METADATA;
  for (int i = 0; i < n_docs; ++i) {
    const int64_t P = (int64_t)cup[i + 1] - cup[i];
    const int64_t L = pad ? (int64_t)cu[i + 1] - cu[i] : P;
    if (P < 0 || L < 0 || L > P) return CP_ERR_METADATA;
    if (strategy == CP_DUAL_CHUNK_SWAP && P % (2 * cp_size)) return CP_ERR_DIVISIBILITY;
  }
  if (total_tokens % cp_size) return CP_ERR_DIVISIBILITY;
  return CP_OK;
}

extern "C" int cp_valid_end(const int32_t* cu, const int32_t* cup, int n_docs, int cp_size,
                            int rank, cp_strategy_t strategy, int pad, int64_t* out) {
  if (!out || !cup || (pad && !cu) || n_docs < 1 || cp_size < 1 || rank < -1 || rank >= cp_size)
    return CP_ERR_INVALID_ARG;
  const int64_t T = cup[n_docs];
  int st = cp_validate_seqlens(cu, cup, n_docs, T, rank < 0 ? 1 : cp_size,
                               rank < 0 ? CP_NO_LOAD_BALANCE : strategy, pad);
  if (st != CP_OK) return st;
  int64_t ve = 0;
  auto real_len = [&](int i) -> int64_t {
    return pad ? (int64_t)cu[i + 1] - cu[i] : (int64_t)cup[i + 1] - cup[i];
  };
  if (rank < 0) {
    for (int i = 0; i < n_docs; ++i)
      if (real_len(i) > 0) ve = std::max<int64_t>(ve, cup[i] + real_len(i));
  } else if (strategy == CP_NO_LOAD_BALANCE) {
    const int64_t s_local = T / cp_size, R0 = rank * s_local, R1 = R0 + s_local;
    for (int i = 0; i < n_docs; ++i) {
      const int64_t a = std::max<int64_t>(cup[i], R0);
      const int64_t e = std::min<int64_t>(cup[i] + real_len(i), R1);
      if (e > a) ve = std::max(ve, e - R0);
    }
  } else {
    int64_t local = 0;
    for (int i = 0; i < n_docs; ++i) {
      const int64_t c = ((int64_t)cup[i + 1] - cup[i]) / (2 * cp_size);
      const int64_t chunks[2] = {rank, 2 * cp_size - 1 - rank};
      for (int q = 0; q < 2; ++q) {
        const int64_t v = std::min(std::max<int64_t>(real_len(i) - chunks[q] * c, 0), c);
        if (v > 0) ve = std::max(ve, local + v);
        local += c;
      }
    }
  }
  *out = ve;
  return CP_OK;
}

extern "C" int cp_device_status(int* status, int reset) {
  if (!status) return CP_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return CP_ERR_CUDA;
  int first = CP_OK;
  const int parts[5] = {cpthd_status_partition(reset), cpthd_status_rows(reset),
                        cpthd_status_attn(reset), cpthd_status_fwd_tc(reset),
                        cpthd_status_bwd_tc(reset)};
  for (int v : parts) {
    if (v == CP_ERR_CUDA) return CP_ERR_CUDA;
    if (first == CP_OK && v != CP_OK) first = v;
  }
  *status = first;
  return CP_OK;
}
