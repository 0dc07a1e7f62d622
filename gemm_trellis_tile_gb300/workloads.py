"""Byte and flop accounting of the trellis workloads (used by the benchmark).

Algorithmic bytes of one layer application at M tokens are what the method must
move: the trellis code words (in * out * bits / 8), the side vectors (rin, rout
fp16 and s_in, s_out fp32: 6 bytes per channel) and the activations read and
written (2 bytes * M * (in + out)).  The fp16 weights the codec avoids are not
counted.  Algorithmic flops are 2 * M * in * out.
"""


def code_bytes(in_features, out_features, bits):
    return in_features * out_features * bits // 8


def side_bytes(in_features, out_features):
    return 6 * (in_features + out_features)


def act_bytes(m, in_features, out_features):
    return 2 * m * (in_features + out_features)


def layer_bytes(m, in_features, out_features, bits):
    return (code_bytes(in_features, out_features, bits) + side_bytes(in_features, out_features)
            + act_bytes(m, in_features, out_features))


def layer_flops(m, in_features, out_features):
    return 2 * m * in_features * out_features


def mlp_layers(hidden, inter, bits):
    """(in, out, bits) of gate, up and down."""
    bg, bu, bd = bits
    return [(hidden, inter, bg), (hidden, inter, bu), (inter, hidden, bd)]


def mlp_bytes(m, hidden, inter, bits):
    return sum(layer_bytes(m, i, o, b) for i, o, b in mlp_layers(hidden, inter, bits))


def gemv_kernel_bytes(m, layers):
    """Bytes the trellis GEMV launches must move for the given (in, out, bits)
    layers: code words plus their fp16-sized activation operands."""
    return sum(code_bytes(i, o, b) + act_bytes(m, i, o) for i, o, b in layers)


def moe_expert_weights(hidden, inter):
    return 3 * hidden * inter
