"""OpPatternKind and the operator table.

TVM "Operator Fusion", Operator Pattern Classification: the kinds are ordered
integers (elementwise 0, broadcast 1, injective 2, commutative reduce 3,
out-elementwise-fusable 4, tuple 7, opaque 8); patterns merge by taking the
maximum.
"""
K_ELEMWISE = 0
K_BROADCAST = 1
K_INJECTIVE = 2
K_COMM_REDUCE = 3
K_OUT_EWISE_FUSABLE = 4
K_TUPLE = 7
K_OPAQUE = 8

# operator -> (pattern kind, allowed operand counts)
OP_TABLE = {
    "add": (K_ELEMWISE, (2, 3)),
    "sub": (K_ELEMWISE, (2,)),
    "mul": (K_ELEMWISE, (2,)),
    "div": (K_ELEMWISE, (2,)),
    "scale": (K_ELEMWISE, (1,)),
    "addc": (K_ELEMWISE, (1,)),
    "relu": (K_ELEMWISE, (1,)),
    "exp": (K_ELEMWISE, (1,)),
    "sigmoid": (K_ELEMWISE, (1,)),
    "tanh": (K_ELEMWISE, (1,)),
    "neg": (K_ELEMWISE, (1,)),
    # bias_add is the page's own example of a broadcast op
    "badd_col": (K_BROADCAST, (2,)),
    "bmul_col": (K_BROADCAST, (2,)),
    "badd_row": (K_BROADCAST, (2,)),
    "bmul_row": (K_BROADCAST, (2,)),
    # transpose reorders axes, so it is injective, not broadcast
    "transpose": (K_INJECTIVE, (1,)),
    "reshape": (K_INJECTIVE, (1,)),
    "rowsum": (K_COMM_REDUCE, (1,)),
    "rowmax": (K_COMM_REDUCE, (1,)),
    "matmul_bf16": (K_OUT_EWISE_FUSABLE, (2,)),
    "opaque_copy": (K_OPAQUE, (1,)),
    # a tuple groups 2-D values of one width (laid out as their rows stacked
    # in order); concat joins a tuple's fields, an injective op
    "tuple": (K_TUPLE, (2, 3, 4)),
    "concat": (K_INJECTIVE, (1,)),
}


def combine(a: int, b: int) -> int:
    """CombinePattern: the more complex of the two."""
    return max(a, b)


def op_kind(op: str) -> int:
    return OP_TABLE[op][0]


def edge_kind(spec, producer_vid: int, consumer_vid: int) -> int:
    """Pattern of the dataflow edge producer -> consumer.

    The edge takes the consumer's kind, except that a broadcast consumer
    reading an operand of its own output shape treats that operand
    elementwise.  Without this, bias_add in the page's conv2d + bias_add +
    relu example would block the phase-0 fusion the page describes.
    """
    c = spec.values[consumer_vid]
    k = op_kind(c.op)
    if k == K_BROADCAST and spec.values[producer_vid].shape == c.shape:
        return K_ELEMWISE
    return k
