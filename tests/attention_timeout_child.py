"""Child process of tests/test_gpu_attention_timeout.py.

Usage: python attention_timeout_child.py <stall-build library> <work dir>

Loads the failure-detection build of the library (its MMA thread stops
issuing at a fixed tile, so the other roles' bounded waits run out) next to
the normal library, runs the sparse MLA attention on the inputs the parent
saved in <work dir> (q.npy as bf16 bits, indices.npy, cache.npy) once with
each, and reports in JSON on stdout: the stall build's status word and
whether it left its outputs untouched; the normal library's outputs go to
<work dir>/out.npy and lse.npy for the parent to compare with the oracle.
"""
import ctypes
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import fp8_quantized_paged_concat_gb300 as kvq  # noqa: E402

SENTINEL = -7.0


def main():
    lib_path, work = sys.argv[1], sys.argv[2]
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    q_bits = np.load(os.path.join(work, "q.npy"))
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(np.load(os.path.join(work, "indices.npy"))).to(dev)
    cache = torch.from_numpy(np.load(os.path.join(work, "cache.npy"))).to(dev)
    scale = float(np.load(os.path.join(work, "scale.npy")))
    T, H = q.shape[0], q.shape[1]

    stall = ctypes.CDLL(lib_path)
    fn = stall.kvq_sparse_mla_attention_nvfp4_ds_mla
    fn.argtypes = kvq._SIGNATURES["kvq_sparse_mla_attention_nvfp4_ds_mla"]
    fn.restype = ctypes.c_int32
    out = torch.full((T, H, 512), SENTINEL, dtype=torch.bfloat16, device=dev)
    lse = torch.full((T, H), SENTINEL, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    rc = fn(q.data_ptr(), q.stride(0), q.stride(1), T, H, idx.data_ptr(), idx.stride(0), idx.shape[1],
            cache.data_ptr(), cache.shape[0], cache.shape[1], cache.stride(0), cache.stride(1),
            ctypes.c_float(scale), out.data_ptr(), out.stride(0), out.stride(1), lse.data_ptr(), lse.stride(0),
            status.data_ptr(), stream)
    torch.cuda.synchronize(dev)
    report = {"rc": int(rc), "status": int(status.item()),
              "out_untouched": bool(torch.all(out == SENTINEL).item()),
              "lse_untouched": bool(torch.all(lse == SENTINEL).item())}

    # the same device and process, the normal library
    status.zero_()
    out2, lse2 = kvq.kvq_sparse_mla_attention_nvfp4_ds_mla(q, idx, cache, scale, status=status)
    torch.cuda.synchronize(dev)
    report["normal_status"] = int(status.item())
    np.save(os.path.join(work, "out.npy"), out2.float().cpu().numpy())
    np.save(os.path.join(work, "lse.npy"), lse2.cpu().numpy())
    print(json.dumps(report))


if __name__ == "__main__":
    main()
