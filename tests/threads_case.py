"""Child process of tests/test_threads_gpu.py: the library's first calls in a
fresh process come from several host threads at once, each on its own CUDA
stream -- verify launches of different shapes (so each thread may be the one
that sets the kernel's shared-memory attribute for its context), a tree
verify, the projection GEMMs and the static-scratch prefill.  Every result
must then be bit-identical to the same work done again, one call after the
other.  Exit status 0 on success; a message on stderr otherwise."""
import sys
import threading

import torch

import gated_deltanet_verify_gb300 as gdn
from tests.gpu_util import dims_of, params_of, upload
from workloads.device import empty_outputs
from workloads.synth import Shape, WORKLOADS, make_inputs, make_parents, make_proj

SHAPES = {
    "layer": WORKLOADS["layer_verify"],
    "t64": Shape("thr_t64", n_slots=1, n_qk_heads=16, n_v_heads=48, d_k=128, d_v=128, n_tokens=64, act="bf16",
                 seed=61),
    "small": Shape("thr_small", n_slots=3, n_qk_heads=4, n_v_heads=8, d_k=64, d_v=64, n_tokens=5, act="f32",
                   seed=62),
    "tree": Shape("thr_tree", n_slots=2, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=9, act="bf16",
                  seed=63),
    "proj": Shape("thr_proj", n_slots=1, n_qk_heads=2, n_v_heads=8, d_k=64, d_v=64, n_tokens=5, act="bf16",
                  seed=64, n_embd=256),
    "prefill": Shape("thr_prefill", n_slots=1, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=130,
                     act="bf16", seed=65),
}


def job(name, stream):
    """One workload on `stream`; returns its device results (the inputs are fresh copies)."""
    shape = SHAPES[name]
    inp = make_inputs(shape)
    d = dims_of(shape)
    sp = stream.cuda_stream
    with torch.cuda.stream(stream):             # the uploads too, so that they are ordered before the calls
        x = upload(inp)
        if name in ("layer", "t64", "small"):
            o = empty_outputs(shape, "cuda")
            gdn.gdn_verify_forward(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                                   x["conv_state"], o["cap_state"], o["cap_conv"], o["out"], None, sp)
            res = {"out": o["out"], "cap": o["cap_state"], "state": x["state"], "conv": x["conv_state"]}
        elif name == "tree":
            par = torch.from_numpy(make_parents(shape, "random")).to("cuda")
            o = empty_outputs(shape, "cuda")
            cap_conv = torch.empty((shape.n_slots, shape.n_tokens, 3, shape.conv_channels), dtype=torch.float32,
                                   device="cuda")
            gdn.gdn_verify_tree(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], par, x["state"],
                                x["conv_state"], o["cap_state"], cap_conv, o["out"], None, sp)
            res = {"out": o["out"], "cap": o["cap_state"], "cap_conv": cap_conv}
        elif name == "proj":
            pr = {k: torch.from_numpy(v).view(torch.bfloat16).to("cuda") for k, v in make_proj(shape).items()}
            w = gdn.proj_weights(shape.n_embd, pr["w_in"], pr["w_out"])
            M = shape.n_slots * shape.n_tokens
            act = torch.empty((M, gdn.gdn_proj_in_ld(d)), dtype=torch.bfloat16, device="cuda")
            y = torch.empty((M, shape.n_embd), dtype=torch.bfloat16, device="cuda")
            gdn.gdn_project_in(d, w, pr["x"], act, None, 0, sp)
            gdn.gdn_project_out(d, w, act[:, :shape.n_v_heads * shape.d_v].contiguous(), y, None, 0, sp)
            res = {"act": act, "y": y}
        else:
            out = torch.empty((shape.n_slots, shape.n_tokens, shape.n_v_heads * shape.d_v), dtype=torch.bfloat16,
                              device="cuda")
            gdn.gdn_prefill_chunked_static(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                                           x["state"], x["conv_state"], out, None, sp)
            res = {"out": out, "state": x["state"], "conv": x["conv_state"]}
    stream.synchronize()
    return res


def main():
    torch.cuda.set_device(0)
    torch.cuda.init()
    # one thread per workload (the static-scratch prefill, whose array is shared per context, in one only)
    names = list(SHAPES)
    got, errors = {}, []
    start = threading.Barrier(len(names))

    def worker(name):
        try:
            s = torch.cuda.Stream()
            start.wait()
            got[name] = job(name, s)
        except Exception as e:          # reported below
            errors.append(f"{name}: {e!r}")

    threads = [threading.Thread(target=worker, args=(n,)) for n in names]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    if errors or len(got) != len(names):
        print("threads failed:", errors, sorted(got), file=sys.stderr)
        return 1
    torch.cuda.synchronize()
    bad = []
    for name in names:
        again = job(name, torch.cuda.Stream())
        for k, v in again.items():
            if not torch.equal(v, got[name][k]):
                bad.append(f"{name}.{k}")
    if bad:
        print("not bit-identical to the sequential rerun:", bad, file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
